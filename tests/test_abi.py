"""Host-side checks of the C ABI (no GPU): the library builds and loads, it
exports every entry point include/vae.h declares, the ctypes mirror of the
chain structs matches the C layout, and argument validation rejects bad
calls before touching the device."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import diffusion_vae_decoder_gb300 as pkg
    if not os.path.exists(pkg.LIB_PATH):
        from diffusion_vae_decoder_gb300 import _build
        _build.build()
    return pkg.load_library()


def test_header_declares_the_five_entry_points():
    import diffusion_vae_decoder_gb300 as pkg
    names = set(pkg.header_symbols())
    for fn in ("vae_conv2d", "vae_groupnorm_silu", "vae_upsample_conv", "vae_mid_attn",
               "vae_decode_chain"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    import diffusion_vae_decoder_gb300 as pkg
    names = pkg.header_symbols()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(names) <= exported


def test_every_header_symbol_has_a_ctypes_signature():
    import diffusion_vae_decoder_gb300 as pkg
    assert set(pkg.header_symbols()) == set(pkg._SIGS)


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "vae.h"
#define P(T) printf(#T " %zu\n", sizeof(T));
#define O(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  P(vae_conv_ref) P(vae_norm_ref) P(vae_resnet_ref) P(vae_attn_ref) P(vae_up_ref)
  P(vae_chain_args) P(vae_prof_record) P(vae_trace_point)
  O(vae_prof_record, flops) O(vae_prof_record, ms)
  O(vae_trace_point, skip) O(vae_trace_point, bytes)
  O(vae_conv_ref, k) O(vae_resnet_ref, shortcut) O(vae_attn_ref, out)
  O(vae_up_ref, resnets) O(vae_up_ref, upsample_conv)
  O(vae_chain_args, eps) O(vae_chain_args, conv_in) O(vae_chain_args, mid_attn)
  O(vae_chain_args, n_ups) O(vae_chain_args, ups) O(vae_chain_args, conv_out)
  O(vae_chain_args, precision) P(vae_causal_decoder_args)
  O(vae_causal_decoder_args, mid) O(vae_causal_decoder_args, ups)
  O(vae_causal_decoder_args, conv_out) O(vae_causal_decoder_args, precision)
  return 0;
}
"""


def test_ctypes_struct_layout_matches_c(tmp_path):
    import diffusion_vae_decoder_gb300 as pkg
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(ln.rsplit(" ", 1) for ln in subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.splitlines())
    m = {"vae_conv_ref": pkg.ConvRef, "vae_norm_ref": pkg.NormRef,
         "vae_resnet_ref": pkg.ResnetRef, "vae_attn_ref": pkg.AttnRef,
         "vae_up_ref": pkg.UpRef, "vae_chain_args": pkg.ChainArgs,
         "vae_prof_record": pkg.ProfRecord, "vae_trace_point": pkg.TracePoint,
         "vae_causal_decoder_args": pkg.CausalDecoderArgs}
    for key, val in got.items():
        if "." in key:
            t, f = key.split(".")
            assert getattr(m[t], f).offset == int(val), key
        else:
            assert ctypes.sizeof(m[key]) == int(val), key


def test_status_strings(lib):
    assert lib.vae_status_string(0) == b"ok"
    assert lib.vae_status_string(-3) == b"workspace too small"
    assert lib.vae_status_string(-99) == b"unknown status"


def test_argument_checks_reject_before_any_launch(lib):
    # null pointers and bad enums are caught on the host; no CUDA call happens
    assert lib.vae_conv2d(None, 1, 32, 8, 8, 0, None, None, 32, 3, None, None, None, None, 0,
                          None, None, 0, None) == -1
    fake = ctypes.c_void_p(16)
    assert lib.vae_conv2d(fake, 1, 32, 8, 8, 7, fake, None, 32, 3, None, None, None, None, 0,
                          fake, fake, 1 << 20, None) == -1
    assert lib.vae_conv2d(fake, 1, 32, 8, 8, 0, fake, None, 32, 5, None, None, None, None, 0,
                          fake, fake, 1 << 20, None) == -2
    assert lib.vae_conv2d(fake, 1, 32, 8, 8, 0, fake, None, 32, 3, None, fake, None, None, 0,
                          fake, fake, 1 << 20, None) == -1
    assert lib.vae_decode_chain(None, fake, 1, 8, 8, fake, fake, 1, None) == -5
    assert lib.vae_chain_destroy(None) == -5
    assert lib.vae_chain_workspace_size(None, 1, 8, 8) == 0
    assert lib.vae_chain_prepare(None, None, None) == -1
    assert lib.vae_chain_profile(None, 1) == -5
    assert lib.vae_kernel_launch_count() == 0
    assert lib.vae_groupnorm_silu(fake, 1, 32, 64, 3, 32, 1e-6, fake, fake, 1, fake, fake,
                                  1 << 20, None) == -1
    assert lib.vae_mid_attn(fake, 1, 48, 4, 4, 0, 16, 1e-6, *([fake] * 11), fake, 1 << 20,
                            None) == -2


def test_unknown_handles_are_rejected_without_being_read(lib):
    """Handles are checked against the registry of live handles, never read
    through: a pointer that vae_chain_prepare did not return (here an address
    that would fault if dereferenced) is refused by every handle entry point."""
    bogus = ctypes.c_void_p(0x10)
    fake = ctypes.c_void_p(16)
    cnt = ctypes.c_int(-1)
    assert lib.vae_chain_destroy(bogus) == -5
    assert lib.vae_decode_chain(bogus, fake, 1, 8, 8, fake, fake, 1, None) == -5
    assert lib.vae_decode_chain_traced(bogus, fake, 1, 8, 8, fake, fake, 1, None, 0, None) == -5
    assert lib.vae_chain_trace_points(bogus, 1, 8, 8, None, 0, ctypes.byref(cnt)) == -5
    assert lib.vae_chain_workspace_size(bogus, 1, 8, 8) == 0
    assert lib.vae_chain_profile(bogus, 1) == -5
    assert lib.vae_chain_profile_read(bogus, None, 0, ctypes.byref(cnt)) == -5


def test_debug_hooks_validate_their_arguments(lib):
    assert lib.vae_debug_inject(2) == -1
    assert lib.vae_debug_inject(0) == 0
    assert lib.vae_debug_fail_allocation(-1) == -1
    assert lib.vae_debug_fail_allocation(0) == 0
    assert lib.vae_debug_set_wait_limit(0) == 0


def test_workspace_sizes_are_positive_and_monotone(lib):
    a = lib.vae_conv2d_workspace_size(1, 128, 64, 64, 0, 128, 3, 0)
    b = lib.vae_conv2d_workspace_size(2, 128, 64, 64, 0, 128, 3, 0)
    assert 0 < a < b
    assert lib.vae_conv2d_workspace_size(1, 128, 64, 64, 1, 128, 3, 0) < a  # NHWC: no staging
    assert lib.vae_upsample_conv_workspace_size(1, 64, 16, 16, 0, 64) > 0
    assert lib.vae_groupnorm_silu_workspace_size(1, 128, 4096, 0, 32) > 0
    assert lib.vae_mid_attn_workspace_size(1, 128, 8, 8, 0) > 128 * 64 * 4
    assert lib.vae_conv3d_causal_workspace_size(1, 32, 3, 8, 8, 0, 32) > 0
    assert lib.vae_conv2d_workspace_size(0, 128, 64, 64, 0, 128, 3, 0) == 0


def test_product_path_refuses_without_library(tmp_path, monkeypatch):
    import diffusion_vae_decoder_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        pkg.load_library(str(tmp_path / "missing.so"))


def test_package_never_imports_the_oracle():
    code = ("import sys; import diffusion_vae_decoder_gb300; "
            "assert 'oracle' not in sys.modules and 'vae_synth' not in sys.modules")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)
