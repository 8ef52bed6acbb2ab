"""GB300 (sm_103a) FLUX-class AutoencoderKL latent decoder.

A thin ctypes binding over the C ABI in ``include/vae.h`` (``libvae.so``).
Every step of the decoder runs in this library's CUDA kernels; this module only
marshals arguments: it takes torch CUDA tensors, allocates outputs and
workspaces through torch, and passes device pointers plus the current stream.
There is no CPU fallback: if the shared library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvae.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "vae.h")

VAE_NCHW = 0
VAE_NHWC = 1
STATUS = {0: "VAE_OK", -1: "VAE_EINVAL", -2: "VAE_EUNSUPPORTED", -3: "VAE_EWORKSPACE",
          -4: "VAE_ECUDA", -5: "VAE_ENOTPREPARED", -6: "VAE_EDEVICE_TIMEOUT", -7: "VAE_ENOMEM"}

_lib = None


class VaeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


# ---------------------------------------------------------------- ctypes mirror of vae.h
_P = ctypes.c_void_p


class ConvRef(ctypes.Structure):
    _fields_ = [("weight", _P), ("bias", _P), ("cout", ctypes.c_int), ("cin", ctypes.c_int),
                ("k", ctypes.c_int)]


class NormRef(ctypes.Structure):
    _fields_ = [("weight", _P), ("bias", _P), ("c", ctypes.c_int)]


class ResnetRef(ctypes.Structure):
    _fields_ = [("norm1", NormRef), ("conv1", ConvRef), ("norm2", NormRef), ("conv2", ConvRef),
                ("shortcut", ConvRef)]


class AttnRef(ctypes.Structure):
    _fields_ = [("norm", NormRef), ("q", ConvRef), ("k", ConvRef), ("v", ConvRef),
                ("out", ConvRef)]


class UpRef(ctypes.Structure):
    _fields_ = [("n_resnets", ctypes.c_int), ("resnets", ctypes.POINTER(ResnetRef)),
                ("upsample_conv", ConvRef)]


class ChainArgs(ctypes.Structure):
    _fields_ = [("latent_channels", ctypes.c_int), ("scaling_factor", ctypes.c_float),
                ("shift_factor", ctypes.c_float), ("groups", ctypes.c_int),
                ("eps", ctypes.c_float), ("conv_in", ConvRef), ("mid_res1", ResnetRef),
                ("mid_attn", AttnRef), ("mid_res2", ResnetRef), ("n_ups", ctypes.c_int),
                ("ups", ctypes.POINTER(UpRef)), ("norm_out", NormRef), ("conv_out", ConvRef),
                ("precision", ctypes.c_int)]


PRECISION_AUTO, PRECISION_TF32, PRECISION_SPLIT_TF32 = 0, 1, 2


class CausalDecoderArgs(ctypes.Structure):
    _fields_ = [("latent_channels", ctypes.c_int), ("scaling_factor", ctypes.c_float),
                ("shift_factor", ctypes.c_float), ("groups", ctypes.c_int),
                ("eps", ctypes.c_float), ("conv_in", ConvRef), ("n_mid", ctypes.c_int),
                ("mid", ctypes.POINTER(ResnetRef)), ("n_ups", ctypes.c_int),
                ("ups", ctypes.POINTER(UpRef)), ("norm_out", NormRef), ("conv_out", ConvRef),
                ("precision", ctypes.c_int)]


class ProfRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("kernels", ctypes.c_int), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double), ("ms", ctypes.c_double)]


PROF_KINDS = {0: "conv3x3", 1: "upsample_conv", 2: "groupnorm", 3: "attention", 4: "layout",
              5: "head", 6: "groupnorm_affine"}


class TracePoint(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("c", ctypes.c_int), ("h", ctypes.c_int),
                ("w", ctypes.c_int), ("input", ctypes.c_int), ("skip", ctypes.c_int),
                ("bytes", ctypes.c_size_t)]


TRACE_KINDS = {0: "latent", 1: "conv", 2: "groupnorm", 3: "resnet", 4: "attention",
               5: "upsample", 6: "rgb"}
INJECT_WITHHOLD_STREAMK_FLAG = 1

_I, _LL, _F, _SZ = ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "vae_conv2d_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "vae_conv2d": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _I, _P, _P, _SZ,
                        _P]),
    "vae_conv2d_pack_bytes": (_SZ, [_I, _I, _I, _I]),
    "vae_conv2d_pack": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _P, _SZ, _P]),
    "vae_conv2d_packed": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _I, _P, _P, _SZ, _P]),
    "vae_upsample_conv_pack_bytes": (_SZ, [_I, _I]),
    "vae_upsample_conv_pack": (_I, [_P, _P, _I, _I, _P, _SZ, _P]),
    "vae_upsample_conv_packed": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "vae_upsample_conv_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "vae_upsample_conv": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _SZ, _P]),
    "vae_groupnorm_silu_workspace_size": (_SZ, [_I, _I, _LL, _I, _I]),
    "vae_groupnorm_silu": (_I, [_P, _I, _I, _LL, _I, _I, _F, _P, _P, _I, _P, _P, _SZ, _P]),
    "vae_groupnorm_silu_noalloc": (_I, [_P, _I, _I, _LL, _I, _I, _F, _P, _P, _I, _P, _P]),
    "vae_mid_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "vae_mid_attn": (_I, [_P, _I, _I, _I, _I, _I, _I, _F] + [_P] * 11 + [_P, _SZ, _P]),
    "vae_conv3d_causal_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "vae_conv3d_causal": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "vae_causal_stack_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "vae_causal_stack": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_P),
                              ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P), _I, _F,
                              _P, _P, _SZ, _P]),
    "vae_chain_prepare": (_I, [ctypes.POINTER(ChainArgs), ctypes.POINTER(_P), _P]),
    "vae_chain_workspace_size": (_SZ, [_P, _I, _I, _I]),
    "vae_decode_chain": (_I, [_P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "vae_chain_destroy": (_I, [_P]),
    "vae_status_string": (ctypes.c_char_p, [_I]),
    "vae_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "vae_num_sms": (_I, []),
    "vae_chain_profile": (_I, [_P, _I]),
    "vae_chain_profile_read": (_I, [_P, ctypes.POINTER(ProfRecord), _I, ctypes.POINTER(_I)]),
    "vae_kernel_launch_count": (_LL, []),
    "vae_chain_trace_points": (_I, [_P, _I, _I, _I, ctypes.POINTER(TracePoint), _I,
                                    ctypes.POINTER(_I)]),
    "vae_decode_chain_traced": (_I, [_P, _P, _I, _I, _I, _P, _P, _SZ, ctypes.POINTER(_P), _I,
                                     _P]),
    "vae_causal_decoder_prepare": (_I, [ctypes.POINTER(CausalDecoderArgs), ctypes.POINTER(_P),
                                        _P]),
    "vae_causal_decoder_workspace_size": (_SZ, [_P, _I, _I, _I, _I]),
    "vae_decode_causal": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "vae_chain_tiled_workspace_size": (_SZ, [_P, _I, _I, _I, _I, _I, _I]),
    "vae_decode_chain_tiled": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "vae_measure_tf32_mma": (_I, [_I, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_float), _P]),
    "vae_debug_set_wait_limit": (_I, [ctypes.c_ulonglong]),
    "vae_debug_inject": (_I, [_I]),
    "vae_debug_fail_allocation": (_I, [_I]),
}


def header_symbols() -> list[str]:
    """Names of every entry point include/vae.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return re.findall(r"^VAE_API\s+[\w\s\*]*?\b(vae_\w+)\s*\(", text, flags=re.M)


def load_library(path: str = LIB_PATH):
    """Load libvae.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn, status):
    if status != 0:
        raise VaeError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name):
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32
            and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    return t


def _ws(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _opt(t, name):
    return None if t is None else _need(t, name)


# ---------------------------------------------------------------- single ops
def vae_conv2d(x, weight, bias=None, residual=None, sc_x=None, sc_w=None, sc_b=None,
               layout=VAE_NCHW, out=None, stream=None):
    lib = load_library()
    _need(x, "x"), _need(weight, "weight")
    bias, residual, sc_x, sc_b = (_opt(bias, "bias"), _opt(residual, "residual"),
                                  _opt(sc_x, "sc_x"), _opt(sc_b, "sc_b"))
    if layout == VAE_NCHW:
        n, cin, h, w = x.shape
    else:
        n, h, w, cin = x.shape
    cout, _, k, _ = weight.shape
    sc_cin = 0
    if sc_w is not None:
        sc_w = _need(sc_w.reshape(sc_w.shape[0], -1).contiguous(), "sc_w")
        sc_cin = sc_w.shape[1]
    shape = (n, cout, h, w) if layout == VAE_NCHW else (n, h, w, cout)
    if out is None:
        import torch
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    ws_bytes = lib.vae_conv2d_workspace_size(n, cin, h, w, layout, cout, k, sc_cin)
    ws = _ws(ws_bytes, x.device)
    _check("vae_conv2d", lib.vae_conv2d(
        _ptr(x), n, cin, h, w, layout, _ptr(weight), _ptr(bias), cout, k, _ptr(residual),
        _ptr(sc_x), _ptr(sc_w), _ptr(sc_b), sc_cin, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


class PackedWeights:
    """A conv's weights packed once on the device (vae_conv2d_pack /
    vae_upsample_conv_pack): the byte buffer and the sizes it was made for."""

    def __init__(self, kind, buf, cout, cin, k, sc_cin):
        self.kind, self.buf = kind, buf
        self.cout, self.cin, self.k, self.sc_cin = cout, cin, k, sc_cin


def vae_conv2d_pack(weight, bias=None, sc_w=None, sc_b=None, stream=None):
    import torch
    lib = load_library()
    _need(weight, "weight")
    bias, sc_b = _opt(bias, "bias"), _opt(sc_b, "sc_b")
    cout, cin, k, _ = weight.shape
    sc_cin = 0
    if sc_w is not None:
        sc_w = _need(sc_w.reshape(sc_w.shape[0], -1).contiguous(), "sc_w")
        sc_cin = sc_w.shape[1]
    nbytes = lib.vae_conv2d_pack_bytes(cout, cin, k, sc_cin)
    buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=weight.device)
    _check("vae_conv2d_pack", lib.vae_conv2d_pack(
        _ptr(weight), _ptr(bias), cout, cin, k, _ptr(sc_w), _ptr(sc_b), sc_cin, _ptr(buf),
        buf.numel(), _stream(stream)))
    return PackedWeights("conv2d", buf, cout, cin, k, sc_cin)


def vae_conv2d_packed(x, pack, residual=None, sc_x=None, layout=VAE_NCHW, out=None, stream=None):
    lib = load_library()
    _need(x, "x")
    residual, sc_x = _opt(residual, "residual"), _opt(sc_x, "sc_x")
    if pack.kind != "conv2d":
        raise TypeError("pack was not made by vae_conv2d_pack")
    if layout == VAE_NCHW:
        n, cin, h, w = x.shape
    else:
        n, h, w, cin = x.shape
    cout, k = pack.cout, pack.k
    shape = (n, cout, h, w) if layout == VAE_NCHW else (n, h, w, cout)
    if out is None:
        import torch
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    ws = _ws(lib.vae_conv2d_workspace_size(n, cin, h, w, layout, cout, k, pack.sc_cin), x.device)
    _check("vae_conv2d_packed", lib.vae_conv2d_packed(
        _ptr(x), n, cin, h, w, layout, _ptr(pack.buf), cout, k, _ptr(residual), _ptr(sc_x),
        pack.sc_cin, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def vae_upsample_conv_pack(weight, bias=None, stream=None):
    import torch
    lib = load_library()
    _need(weight, "weight")
    bias = _opt(bias, "bias")
    cout, cin = weight.shape[0], weight.shape[1]
    nbytes = lib.vae_upsample_conv_pack_bytes(cout, cin)
    buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=weight.device)
    _check("vae_upsample_conv_pack", lib.vae_upsample_conv_pack(
        _ptr(weight), _ptr(bias), cout, cin, _ptr(buf), buf.numel(), _stream(stream)))
    return PackedWeights("upsample_conv", buf, cout, cin, 3, 0)


def vae_upsample_conv_packed(x, pack, layout=VAE_NCHW, out=None, stream=None):
    lib = load_library()
    _need(x, "x")
    if pack.kind != "upsample_conv":
        raise TypeError("pack was not made by vae_upsample_conv_pack")
    if layout == VAE_NCHW:
        n, cin, h, w = x.shape
    else:
        n, h, w, cin = x.shape
    cout = pack.cout
    shape = (n, cout, 2 * h, 2 * w) if layout == VAE_NCHW else (n, 2 * h, 2 * w, cout)
    if out is None:
        import torch
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    ws = _ws(lib.vae_upsample_conv_workspace_size(n, cin, h, w, layout, cout), x.device)
    _check("vae_upsample_conv_packed", lib.vae_upsample_conv_packed(
        _ptr(x), n, cin, h, w, layout, _ptr(pack.buf), cout, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def vae_upsample_conv(x, weight, bias=None, layout=VAE_NCHW, out=None, stream=None):
    lib = load_library()
    _need(x, "x"), _need(weight, "weight")
    bias = _opt(bias, "bias")
    if layout == VAE_NCHW:
        n, cin, h, w = x.shape
    else:
        n, h, w, cin = x.shape
    cout = weight.shape[0]
    shape = (n, cout, 2 * h, 2 * w) if layout == VAE_NCHW else (n, 2 * h, 2 * w, cout)
    if out is None:
        import torch
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    ws = _ws(lib.vae_upsample_conv_workspace_size(n, cin, h, w, layout, cout), x.device)
    _check("vae_upsample_conv", lib.vae_upsample_conv(
        _ptr(x), n, cin, h, w, layout, _ptr(weight), _ptr(bias), cout, _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def vae_groupnorm_silu(x, gamma, beta, groups=32, eps=1e-6, apply_silu=True, layout=VAE_NCHW,
                       out=None, stream=None):
    lib = load_library()
    _need(x, "x"), _need(gamma, "gamma"), _need(beta, "beta")
    n = x.shape[0]
    if layout == VAE_NCHW:
        c = x.shape[1]
        spatial = x.numel() // (n * c)
    else:
        c = x.shape[-1]
        spatial = x.numel() // (n * c)
    if out is None:
        import torch
        out = torch.empty_like(x)
    ws = _ws(lib.vae_groupnorm_silu_workspace_size(n, c, spatial, layout, groups), x.device)
    _check("vae_groupnorm_silu", lib.vae_groupnorm_silu(
        _ptr(x), n, c, spatial, layout, groups, eps, _ptr(gamma), _ptr(beta), int(apply_silu),
        _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def vae_groupnorm_silu_noalloc(x, gamma, beta, groups=32, eps=1e-6, apply_silu=True,
                               layout=VAE_NCHW, out=None, stream=None):
    """GroupNorm(+SiLU) whose scratch is a fixed array inside the library (no
    workspace); for callers that must not allocate device memory."""
    lib = load_library()
    _need(x, "x"), _need(gamma, "gamma"), _need(beta, "beta")
    n = x.shape[0]
    c = x.shape[1] if layout == VAE_NCHW else x.shape[-1]
    spatial = x.numel() // (n * c)
    if out is None:
        import torch
        out = torch.empty_like(x)
    _check("vae_groupnorm_silu_noalloc", lib.vae_groupnorm_silu_noalloc(
        _ptr(x), n, c, spatial, layout, groups, eps, _ptr(gamma), _ptr(beta), int(apply_silu),
        _ptr(out), _stream(stream)))
    return out


def vae_mid_attn(x, p, groups=32, eps=1e-6, layout=VAE_NCHW, out=None, stream=None):
    """``p``: dict with group_norm / to_q / to_k / to_v / to_out -> (weight, bias)."""
    lib = load_library()
    _need(x, "x")
    if layout == VAE_NCHW:
        n, c, h, w = x.shape
    else:
        n, h, w, c = x.shape
    ptrs = []
    for key in ("group_norm", "to_q", "to_k", "to_v", "to_out"):
        wt, b = p[key]
        ptrs += [_ptr(_need(wt, key)), _ptr(_need(b, key))]
    if out is None:
        import torch
        out = torch.empty_like(x)
    ws = _ws(lib.vae_mid_attn_workspace_size(n, c, h, w, layout), x.device)
    _check("vae_mid_attn", lib.vae_mid_attn(
        _ptr(x), n, c, h, w, layout, groups, eps, *ptrs, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def vae_conv3d_causal(x, weight, bias=None, residual=None, layout=VAE_NCHW, out=None,
                      stream=None):
    lib = load_library()
    _need(x, "x"), _need(weight, "weight")
    bias, residual = _opt(bias, "bias"), _opt(residual, "residual")
    if layout == VAE_NCHW:
        n, cin, t, h, w = x.shape
    else:
        n, t, h, w, cin = x.shape
    cout = weight.shape[0]
    shape = (n, cout, t, h, w) if layout == VAE_NCHW else (n, t, h, w, cout)
    if out is None:
        import torch
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    ws = _ws(lib.vae_conv3d_causal_workspace_size(n, cin, t, h, w, layout, cout), x.device)
    _check("vae_conv3d_causal", lib.vae_conv3d_causal(
        _ptr(x), n, cin, t, h, w, layout, _ptr(weight), _ptr(bias), cout, _ptr(residual),
        _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def vae_kernel_launch_count():
    return load_library().vae_kernel_launch_count()


def vae_causal_stack(x, layers, groups=32, eps=1e-6, layout=VAE_NCHW, out=None, stream=None):
    """``layers``: list of dicts with weight [c,c,3,3,3], bias, gn_weight, gn_bias (CUDA)."""
    lib = load_library()
    _need(x, "x")
    if layout == VAE_NCHW:
        n, c, t, h, w = x.shape
    else:
        n, t, h, w, c = x.shape
    L = len(layers)
    arr = lambda key: (_P * L)(*[_need(d[key], key).data_ptr() for d in layers])  # noqa: E731
    if out is None:
        import torch
        out = torch.empty_like(x)
    ws = _ws(lib.vae_causal_stack_workspace_size(n, c, t, h, w, layout, L), x.device)
    _check("vae_causal_stack", lib.vae_causal_stack(
        _ptr(x), n, c, t, h, w, layout, L, arr("weight"), arr("bias"), arr("gn_weight"),
        arr("gn_bias"), groups, eps, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def vae_measure_tf32_mma(iters, stream=None):
    """(TFLOP/s, ms, flops) of the tensor-pipe TF32 MMA loop (vae_measure_tf32_mma)."""
    flops, ms = ctypes.c_double(0), ctypes.c_float(0)
    _check("vae_measure_tf32_mma", load_library().vae_measure_tf32_mma(
        int(iters), ctypes.byref(flops), ctypes.byref(ms), _stream(stream)))
    return flops.value / (ms.value / 1e3) / 1e12, ms.value, flops.value


def vae_debug_set_wait_limit(ns):
    _check("vae_debug_set_wait_limit", load_library().vae_debug_set_wait_limit(int(ns)))


def vae_debug_inject(bits):
    _check("vae_debug_inject", load_library().vae_debug_inject(int(bits)))


def vae_debug_fail_allocation(nth):
    _check("vae_debug_fail_allocation", load_library().vae_debug_fail_allocation(int(nth)))


def vae_device_error(stream=None):
    lib = load_library()
    code = ctypes.c_int(0)
    _check("vae_device_error", lib.vae_device_error(_stream(stream), ctypes.byref(code)))
    return code.value


# ---------------------------------------------------------------- the chain
def _conv_ref(weights, name, keep):
    w = weights.get(name + ".weight")
    if w is None:
        return ConvRef()
    import numpy as np
    w = np.ascontiguousarray(w, dtype=np.float32)
    b = np.ascontiguousarray(weights[name + ".bias"], dtype=np.float32)
    keep += [w, b]
    return ConvRef(w.ctypes.data, b.ctypes.data, w.shape[0], w.shape[1],
                   w.shape[2] if w.ndim == 4 else 1)


def _norm_ref(weights, name, keep):
    import numpy as np
    g = np.ascontiguousarray(weights[name + ".weight"], dtype=np.float32)
    b = np.ascontiguousarray(weights[name + ".bias"], dtype=np.float32)
    keep += [g, b]
    return NormRef(g.ctypes.data, b.ctypes.data, g.shape[0])


def _resnet_ref(weights, pre, keep):
    return ResnetRef(_norm_ref(weights, pre + ".norm1", keep), _conv_ref(weights, pre + ".conv1", keep),
                     _norm_ref(weights, pre + ".norm2", keep), _conv_ref(weights, pre + ".conv2", keep),
                     _conv_ref(weights, pre + ".conv_shortcut", keep))


class VaeChain:
    """Prepared decoder (vae_chain_prepare / vae_decode_chain / vae_chain_destroy).

    ``weights`` maps diffusers-style names (conv_in.weight, mid.resnets.0...,
    mid.attentions.0.to_q.weight, up_blocks.{i}.resnets.{j}..., ...,
    conv_norm_out.weight, conv_out.weight) to host float32 arrays.
    ``precision``: PRECISION_AUTO (split-TF32 products for decodes with little
    conv work, TF32 otherwise), PRECISION_TF32 or PRECISION_SPLIT_TF32."""

    def __init__(self, weights, n_up_blocks, resnets_per_block=3, latent_channels=16,
                 scaling_factor=0.3611, shift_factor=0.1159, groups=32, eps=1e-6, stream=None,
                 precision=PRECISION_AUTO):
        lib = load_library()
        keep = []
        ups = []
        self._res_arrays = []
        for i in range(n_up_blocks):
            res = (ResnetRef * resnets_per_block)(*[
                _resnet_ref(weights, f"up_blocks.{i}.resnets.{j}", keep)
                for j in range(resnets_per_block)])
            self._res_arrays.append(res)
            ups.append(UpRef(resnets_per_block, res,
                             _conv_ref(weights, f"up_blocks.{i}.upsamplers.0.conv", keep)))
        ups_arr = (UpRef * max(1, n_up_blocks))(*ups)
        a = "mid.attentions.0"
        attn = AttnRef(_norm_ref(weights, a + ".group_norm", keep),
                       *[_conv_ref(weights, f"{a}.{p}", keep)
                         for p in ("to_q", "to_k", "to_v", "to_out")])
        for r in (attn.q, attn.k, attn.v, attn.out):
            r.k = 1
        args = ChainArgs(latent_channels, scaling_factor, shift_factor, groups, eps,
                         _conv_ref(weights, "conv_in", keep),
                         _resnet_ref(weights, "mid.resnets.0", keep), attn,
                         _resnet_ref(weights, "mid.resnets.1", keep), n_up_blocks, ups_arr,
                         _norm_ref(weights, "conv_norm_out", keep),
                         _conv_ref(weights, "conv_out", keep), int(precision))
        h = ctypes.c_void_p()
        _check("vae_chain_prepare", lib.vae_chain_prepare(ctypes.byref(args), ctypes.byref(h),
                                                          _stream(stream)))
        self.handle = h
        self.latent_channels = latent_channels
        self.out_channels = weights["conv_out.weight"].shape[0]
        self.up_factor = 2 ** sum(1 for i in range(n_up_blocks)
                                  if f"up_blocks.{i}.upsamplers.0.conv.weight" in weights)

    def workspace_size(self, n, h, w):
        return load_library().vae_chain_workspace_size(self.handle, n, h, w)

    def decode(self, z, out=None, ws=None, stream=None):
        lib = load_library()
        _need(z, "z")
        n, c, h, w = z.shape
        if out is None:
            import torch
            f = self.up_factor
            out = torch.empty((n, self.out_channels, f * h, f * w), dtype=torch.float32,
                              device=z.device)
        if ws is None:
            ws = _ws(self.workspace_size(n, h, w), z.device)
        _check("vae_decode_chain", lib.vae_decode_chain(
            self.handle, _ptr(z), n, h, w, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
        return out

    def decode_tiled(self, z, tile=512, min_overlap=64, tiles_per_batch=0, out=None, ws=None,
                     stream=None):
        """vae_decode_chain_tiled: decode in overlapping tiles of ``tile``
        output pixels, cross-faded over their overlaps."""
        lib = load_library()
        _need(z, "z")
        n, c, h, w = z.shape
        if out is None:
            import torch
            f = self.up_factor
            out = torch.empty((n, self.out_channels, f * h, f * w), dtype=torch.float32,
                              device=z.device)
        if ws is None:
            nb = lib.vae_chain_tiled_workspace_size(self.handle, n, h, w, tile, min_overlap,
                                                    tiles_per_batch)
            if nb == 0:
                raise VaeError("vae_chain_tiled_workspace_size", -1)
            ws = _ws(nb, z.device)
        _check("vae_decode_chain_tiled", lib.vae_decode_chain_tiled(
            self.handle, _ptr(z), n, h, w, tile, min_overlap, tiles_per_batch, _ptr(out),
            _ptr(ws), ws.numel(), _stream(stream)))
        return out

    def trace_points(self, n, h, w):
        """The decode's trace points (vae_chain_trace_points) as dicts."""
        lib = load_library()
        cnt = ctypes.c_int(0)
        _check("vae_chain_trace_points", lib.vae_chain_trace_points(
            self.handle, n, h, w, None, 0, ctypes.byref(cnt)))
        arr = (TracePoint * max(1, cnt.value))()
        _check("vae_chain_trace_points", lib.vae_chain_trace_points(
            self.handle, n, h, w, arr, cnt.value, ctypes.byref(cnt)))
        return [dict(kind=TRACE_KINDS[p.kind], c=p.c, h=p.h, w=p.w, input=p.input, skip=p.skip,
                     bytes=p.bytes) for p in arr[:cnt.value]]

    def decode_traced(self, z, trace, out=None, ws=None, stream=None):
        """vae_decode_chain_traced: ``trace`` is a list with one CUDA tensor
        (or None) per trace point, receiving that step's output."""
        lib = load_library()
        _need(z, "z")
        n, c, h, w = z.shape
        if out is None:
            import torch
            f = self.up_factor
            out = torch.empty((n, self.out_channels, f * h, f * w), dtype=torch.float32,
                              device=z.device)
        if ws is None:
            ws = _ws(self.workspace_size(n, h, w), z.device)
        bufs = (_P * max(1, len(trace)))(*[None if t is None else t.data_ptr() for t in trace])
        _check("vae_decode_chain_traced", lib.vae_decode_chain_traced(
            self.handle, _ptr(z), n, h, w, _ptr(out), _ptr(ws), ws.numel(), bufs, len(trace),
            _stream(stream)))
        return out

    def capture_graph(self, z, out, ws):
        """Capture one vae_decode_chain call on fixed buffers into a CUDA graph
        (the chain neither synchronises nor allocates); replay() re-runs the
        whole decode with one launch. Make one eager decode first."""
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.decode(z, out=out, ws=ws)
        return g

    def profile(self, enable=True):
        _check("vae_chain_profile", load_library().vae_chain_profile(self.handle, int(enable)))

    def profile_read(self):
        """Per-step records of the profiled decodes (synchronises their events)."""
        lib = load_library()
        cnt = ctypes.c_int(0)
        _check("vae_chain_profile_read", lib.vae_chain_profile_read(self.handle, None, 0,
                                                                    ctypes.byref(cnt)))
        arr = (ProfRecord * max(1, cnt.value))()
        _check("vae_chain_profile_read", lib.vae_chain_profile_read(self.handle, arr, cnt.value,
                                                                    ctypes.byref(cnt)))
        return [dict(kind=PROF_KINDS.get(r.kind, r.kind), kernels=r.kernels, flops=r.flops,
                     bytes=r.bytes, ms=r.ms) for r in arr[:cnt.value]]

    def close(self):
        if getattr(self, "handle", None):
            _check("vae_chain_destroy", load_library().vae_chain_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class VaeCausalDecoder:
    """Prepared 3-D causal decoder (vae_causal_decoder_prepare /
    vae_decode_causal / vae_chain_destroy). ``weights`` as
    vae_synth.make_causal_decoder_weights names them: conv weights
    [cout, cin, 3, 3, 3], 1x1x1 shortcuts [cout, cin, 1, 1]."""

    def __init__(self, weights, n_up_blocks, n_mid=2, resnets_per_block=2, latent_channels=16,
                 scaling_factor=0.3611, shift_factor=0.1159, groups=32, eps=1e-6, stream=None,
                 precision=PRECISION_AUTO):
        lib = load_library()
        keep = []

        def conv(name):
            r = _conv_ref(weights, name, keep)
            if name + ".weight" in weights and weights[name + ".weight"].ndim == 5:
                r.k = 3
            return r

        def res(pre):
            return ResnetRef(_norm_ref(weights, pre + ".norm1", keep), conv(pre + ".conv1"),
                             _norm_ref(weights, pre + ".norm2", keep), conv(pre + ".conv2"),
                             _conv_ref(weights, pre + ".conv_shortcut", keep))

        mid = (ResnetRef * max(1, n_mid))(*[res(f"mid.resnets.{m}") for m in range(n_mid)])
        ups, self._res_arrays = [], [mid]
        for i in range(n_up_blocks):
            arr = (ResnetRef * resnets_per_block)(*[
                res(f"up_blocks.{i}.resnets.{j}") for j in range(resnets_per_block)])
            self._res_arrays.append(arr)
            ups.append(UpRef(resnets_per_block, arr, conv(f"up_blocks.{i}.upsamplers.0.conv")))
        ups_arr = (UpRef * max(1, n_up_blocks))(*ups)
        args = CausalDecoderArgs(latent_channels, scaling_factor, shift_factor, groups, eps,
                                 conv("conv_in"), n_mid, mid, n_up_blocks, ups_arr,
                                 _norm_ref(weights, "conv_norm_out", keep), conv("conv_out"),
                                 int(precision))
        h = ctypes.c_void_p()
        _check("vae_causal_decoder_prepare", lib.vae_causal_decoder_prepare(
            ctypes.byref(args), ctypes.byref(h), _stream(stream)))
        self.handle = h
        self.out_channels = weights["conv_out.weight"].shape[0]
        self.up_factor = 2 ** sum(1 for i in range(n_up_blocks)
                                  if f"up_blocks.{i}.upsamplers.0.conv.weight" in weights)

    def workspace_size(self, n, t, h, w):
        return load_library().vae_causal_decoder_workspace_size(self.handle, n, t, h, w)

    def decode(self, z, out=None, ws=None, stream=None):
        lib = load_library()
        _need(z, "z")
        n, c, t, h, w = z.shape
        if out is None:
            import torch
            f = self.up_factor
            out = torch.empty((n, self.out_channels, t, f * h, f * w), dtype=torch.float32,
                              device=z.device)
        if ws is None:
            ws = _ws(self.workspace_size(n, t, h, w), z.device)
        _check("vae_decode_causal", lib.vae_decode_causal(
            self.handle, _ptr(z), n, t, h, w, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
        return out

    def close(self):
        if getattr(self, "handle", None):
            _check("vae_chain_destroy", load_library().vae_chain_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
