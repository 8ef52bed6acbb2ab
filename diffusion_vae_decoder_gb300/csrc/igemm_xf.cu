// igemm_xf.cu -- the operand-transform instantiations of the implicit-GEMM
// kernel (igemm_kernel.cuh, Cfg XF): four more warps rewrite each landed A
// buffer in shared memory before the MMAs read it.
//   xf 1: GroupNorm (+SiLU) of a 3x3 conv's halo-staged input, so the
//         normalised activation never goes through HBM (the resnet's
//         norm -> conv pairs);
//   xf 2: the row softmax of an attention score stage, with the row
//         statistics gathered by the score GEMM's epilogue, so the
//         probabilities never go through HBM (P.V);
//   xf 3: the conv's A operand, the GroupNorm+SiLU of the layer's input,
//         written by those warps a few rows ahead of the tiles that read it,
//         so the separate normalisation pass overlaps the conv.
// Kept in a translation unit of its own so it compiles in parallel.
#include "igemm_kernel.cuh"

namespace vae {
namespace igk {

int launch_xf(int xf, int mode, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
              const CUtensorMap &ts, const CUtensorMap &to, const CUtensorMap &tr,
              const KParams &kp, cudaStream_t s) {
  if (xf == 3) {
    if (mode == 4) return launch_typed<128, 4, 2, false, false, 3>(ta, tb, ts, to, tr, kp, s);
    if (mode == 3)
      return pair ? launch_typed<256, 3, 1, true, false, 3>(ta, tb, ts, to, tr, kp, s)
                  : launch_typed<256, 3, 1, false, false, 3>(ta, tb, ts, to, tr, kp, s);
    return VAE_EINVAL;
  }
  if (xf == 1)
    return pair ? launch_typed<256, 3, 1, true, false, 1>(ta, tb, ts, to, tr, kp, s)
                : launch_typed<256, 3, 1, false, false, 1>(ta, tb, ts, to, tr, kp, s);
  if (xf == 2)
    return pair ? launch_typed<256, 2, 1, true, false, 2>(ta, tb, ts, to, tr, kp, s)
                : launch_typed<256, 2, 1, false, false, 2>(ta, tb, ts, to, tr, kp, s);
  return VAE_EINVAL;
}

}  // namespace igk
}  // namespace vae
