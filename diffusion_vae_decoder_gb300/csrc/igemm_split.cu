// igemm_split.cu -- the split-TF32 instantiations of the implicit-GEMM kernel
// (igemm_kernel.cuh, Cfg SPLIT): every product a * b is formed as
// a_hi b_hi + a_lo b_hi + a_hi b_lo with each part rounded to TF32, on FP32
// operands, for about FP32 accuracy at three times the MMA work. Kept in a
// translation unit of its own so the two sets of kernels compile in parallel.
#include "igemm_kernel.cuh"

namespace vae {
namespace igk {

namespace {

template <int MODE>
int launch_split_mode(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                      const CUtensorMap &ts, const CUtensorMap &to, const CUtensorMap &tr,
                      const KParams &kp, cudaStream_t s) {
  switch (bn) {
    case 256: return launch_typed<256, MODE, 1, false, true>(ta, tb, ts, to, tr, kp, s);
    case 128:
      return MODE != 2 ? launch_typed<128, MODE, 2, false, true>(ta, tb, ts, to, tr, kp, s)
                       : launch_typed<128, MODE, 1, false, true>(ta, tb, ts, to, tr, kp, s);
    case 64: return launch_typed<64, MODE, 1, false, true>(ta, tb, ts, to, tr, kp, s);
    case 32: return launch_typed<32, MODE, 1, false, true>(ta, tb, ts, to, tr, kp, s);
    default: return launch_typed<16, MODE, 1, false, true>(ta, tb, ts, to, tr, kp, s);
  }
}

}  // namespace

int launch_split(int mode, int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                 const CUtensorMap &ts, const CUtensorMap &to, const CUtensorMap &tr,
                 const KParams &kp, cudaStream_t s) {
  switch (mode) {
    case 0: return launch_split_mode<0>(bn, ta, tb, ts, to, tr, kp, s);
    case 1: return launch_split_mode<1>(bn, ta, tb, ts, to, tr, kp, s);
    case 2: return launch_split_mode<2>(bn, ta, tb, ts, to, tr, kp, s);
    default: return VAE_EINVAL;
  }
}

}  // namespace igk
}  // namespace vae
