"""Python binding of libpisa.so (ctypes). Argument marshalling only: every
step of the attention path runs in the library's CUDA kernels. PyTorch
supplies device memory and the current CUDA stream.

The calls mirror include/pisa.h:
  block_stats(q, k, v)                 -> qbar, kbar, vsum[, hmat]
  route(qbar, kbar, scale, topk, band) -> idx, cnt
  forward(q, k, v, idx, cnt, scale)    -> out
and ``piecewise_sparse_attention`` chains them.
"""

from __future__ import annotations

import ctypes
import math
import threading
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libpisa.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK = range(6)
F32, BF16 = 0, 1
NORM_SPECTRAL, NORM_FROBENIUS = 0, 1
BLOCK = 64

EXPORTED = ("pisa_block_stats", "pisa_route", "pisa_forward", "pisa_status_string",
            "pisa_version", "pisa_last_error", "pisa_selftest_tc", "pisa_global_first_order",
            "pisa_forward_hybrid", "pisa_forward_hybrid_workspace_size",
            "pisa_forward_hybrid_static", "pisa_forward_hybrid_static_capacity",
            "pisa_block_heterogeneity", "pisa_route_covariance", "pisa_second_order_spread",
            "pisa_forward_second_order", "pisa_route_ex", "pisa_morton_permutation",
            "pisa_reorder_heads", "pisa_restore_heads", "pisa_attention_host",
            "pisa_attention_host_workspace_size")


class PisaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {status_string(code)} (status {code})"
        if code == ERR_CUDA:
            msg += f": {last_error()}"
        super().__init__(msg)


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libpisa.so; raises if it has not been built (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.pisa_block_stats.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, vp]
    L.pisa_route.argtypes = [vp, vp, i32, i32, i32, f32, i32, i32, vp, vp, i32, vp, vp]
    L.pisa_forward.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, i32, vp, i32, vp, vp]
    L.pisa_selftest_tc.argtypes = [vp, vp, vp, vp, i32, vp, vp]
    L.pisa_global_first_order.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    L.pisa_forward_hybrid.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp,
                                      i32, vp, i32, vp, ctypes.c_size_t, vp, vp]
    L.pisa_forward_hybrid_workspace_size.argtypes = [i32, i32, i32, i32]
    L.pisa_forward_hybrid_workspace_size.restype = ctypes.c_size_t
    L.pisa_forward_hybrid_static.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp,
                                             vp, vp, i32, vp, i32, vp, vp]
    L.pisa_forward_hybrid_static.restype = i32
    L.pisa_block_heterogeneity.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp]
    L.pisa_route_covariance.argtypes = [vp, vp, vp, f32, i32, i32, i32, f32, i32, i32, vp, vp, i32,
                                        vp, vp]
    L.pisa_second_order_spread.argtypes = [vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp,
                                           vp, vp, vp]
    L.pisa_forward_second_order.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, i32,
                                            vp, vp, i32, vp, vp]
    L.pisa_route_ex.argtypes = [vp, vp, vp, f32, vp, i32, i32, i32, f32, i32, i32, i32, vp, vp, i32,
                                vp, vp]
    L.pisa_morton_permutation.argtypes = [i32, i32, i32, i32, vp, vp, vp]
    L.pisa_reorder_heads.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.pisa_restore_heads.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.pisa_forward_hybrid_static_capacity.argtypes = []
    L.pisa_forward_hybrid_static_capacity.restype = ctypes.c_size_t
    L.pisa_attention_host.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, vp, i32,
                                      i32, i32, vp, ctypes.c_size_t, vp, vp]
    L.pisa_attention_host.restype = i32
    L.pisa_attention_host_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    L.pisa_attention_host_workspace_size.restype = ctypes.c_size_t
    for name in ("pisa_block_stats", "pisa_route", "pisa_forward", "pisa_selftest_tc", "pisa_version",
                 "pisa_global_first_order", "pisa_forward_hybrid", "pisa_block_heterogeneity",
                 "pisa_route_covariance", "pisa_second_order_spread", "pisa_forward_second_order",
                 "pisa_route_ex", "pisa_morton_permutation", "pisa_reorder_heads",
                 "pisa_restore_heads"):
        getattr(L, name).restype = i32
    L.pisa_status_string.argtypes = [i32]
    L.pisa_status_string.restype = ctypes.c_char_p
    L.pisa_last_error.argtypes = []
    L.pisa_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().pisa_status_string(int(code)).decode()


def last_error() -> str:
    """The library's description of its last CUDA failure on this thread."""
    return load().pisa_last_error().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dt}")


def _check(rc, where):
    if rc != OK:
        raise PisaError(rc, where)


def _qkv(q, k, v):
    if q.dim() != 3 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share the shape [heads, n, d]")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    return [t.contiguous() for t in (q, k, v)]


def _check_out(out, shape, device):
    """A caller-given output must be exactly what the kernels write: a
    contiguous bf16 or float32 CUDA tensor of ``shape`` on ``device`` (the C
    side cannot see the buffer's size, so a short or strided one would be
    overrun)."""
    if not isinstance(out, torch.Tensor) or not out.is_cuda or out.device != device:
        raise ValueError(f"out must be a CUDA tensor on {device}")
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {tuple(shape)}")
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"out must be bfloat16 or float32, not {out.dtype}")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")


def _require(name, t, shape, dtype, device):
    """An input used as it is: right shape, dtype and device, and already
    contiguous (no copy is made)."""
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (this call makes no copy)")


def new_status(device=None):
    """Zeroed device status word for the optional ``dev_status`` argument."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(status):
    """Synchronise and raise if a kernel stored an error in ``status``."""
    code = int(status.item())
    if code != OK:
        raise PisaError(code, "device")


def block_stats(q, k, v, *, with_vsum=True, with_h=False, h_dtype=torch.float32, status=None,
                stream=None):
    """Per-block qbar, kbar (means) and optionally Vhat (sum) and H."""
    q, k, v = _qkv(q, k, v)
    H, n, d = q.shape
    nb = -(-n // BLOCK)
    f = dict(device=q.device, dtype=torch.float32)
    qbar = torch.empty(H, nb, d, **f)
    kbar = torch.empty(H, nb, d, **f)
    vsum = torch.empty(H, nb, d, **f) if with_vsum else None
    hmat = torch.empty(H, nb, d, d, device=q.device, dtype=h_dtype) if with_h else None
    rc = load().pisa_block_stats(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n, d, BLOCK,
                                 _ptr(qbar), _ptr(kbar), _ptr(vsum), _ptr(hmat),
                                 _dtype_code(h_dtype), _ptr(status), _stream(stream))
    _check(rc, "pisa_block_stats")
    return qbar, kbar, vsum, hmat


def global_first_order(k, v, kbar, vsum, *, status=None, stream=None):
    """Hbar [heads, d, d] = mean over blocks of H_j (hybrid approximation)."""
    _, k, v = _qkv(k, k, v)
    H, n, d = k.shape
    hbar = torch.empty(H, d, d, device=k.device, dtype=torch.float32)
    rc = load().pisa_global_first_order(_ptr(k), _ptr(v), _dtype_code(k.dtype), H, n, d, BLOCK,
                                        _ptr(kbar.contiguous()), _ptr(vsum.contiguous()),
                                        _ptr(hbar), _ptr(status), _stream(stream))
    _check(rc, "pisa_global_first_order")
    return hbar


def max_sel(nb: int, topk: int, band: int) -> int:
    return min(nb, topk + 2 * band + 1)


def route(qbar, kbar, scale: float, topk: int, band: int = 1, *, status=None, stream=None):
    """Critical block list per query block: idx [H, nb, max_sel] (ascending,
    -1 padded) and cnt [H, nb]."""
    if qbar.shape != kbar.shape or qbar.dim() != 3:
        raise ValueError("qbar, kbar must be [heads, nb, d]")
    qbar, kbar = qbar.contiguous(), kbar.contiguous()
    H, nb, d = qbar.shape
    ms = max_sel(nb, topk, band)
    idx = torch.empty(H, nb, ms, device=qbar.device, dtype=torch.int32)
    cnt = torch.empty(H, nb, device=qbar.device, dtype=torch.int32)
    rc = load().pisa_route(_ptr(qbar), _ptr(kbar), H, nb, d, float(scale), int(topk), int(band),
                           _ptr(idx), _ptr(cnt), ms, _ptr(status), _stream(stream))
    _check(rc, "pisa_route")
    return idx, cnt


def block_heterogeneity(k, v, kbar, hbar, *, norm="spectral", status=None, stream=None):
    """M [heads, nb] = ||H_j - Hbar|| (spectral or Frobenius) per block."""
    _, k, v = _qkv(k, k, v)
    H, n, d = k.shape
    nb = -(-n // BLOCK)
    code = {"spectral": NORM_SPECTRAL, "frobenius": NORM_FROBENIUS}[norm]
    mnorm = torch.empty(H, nb, device=k.device, dtype=torch.float32)
    rc = load().pisa_block_heterogeneity(_ptr(k), _ptr(v), _dtype_code(k.dtype), H, n, d, BLOCK,
                                         _ptr(kbar.contiguous()), _ptr(hbar.contiguous()), code,
                                         _ptr(mnorm), _ptr(status), _stream(stream))
    _check(rc, "pisa_block_heterogeneity")
    return mnorm


def route_covariance(qbar, kbar, mnorm, scale: float, topk: int, band: int = 1, *,
                     eps: float = 1e-6, status=None, stream=None):
    """Covariance-aware critical block lists (score s qbar.kbar + log(M + eps)):
    idx [H, nb, max_sel] (ascending, -1 padded) and cnt [H, nb]."""
    if qbar.shape != kbar.shape or qbar.dim() != 3 or mnorm.shape != qbar.shape[:2]:
        raise ValueError("qbar, kbar must be [heads, nb, d] and mnorm [heads, nb]")
    qbar, kbar, mnorm = qbar.contiguous(), kbar.contiguous(), mnorm.contiguous()
    H, nb, d = qbar.shape
    ms = max_sel(nb, topk, band)
    idx = torch.empty(H, nb, ms, device=qbar.device, dtype=torch.int32)
    cnt = torch.empty(H, nb, device=qbar.device, dtype=torch.int32)
    rc = load().pisa_route_covariance(_ptr(qbar), _ptr(kbar), _ptr(mnorm), float(eps), H, nb, d,
                                      float(scale), int(topk), int(band), _ptr(idx), _ptr(cnt),
                                      ms, _ptr(status), _stream(stream))
    _check(rc, "pisa_route_covariance")
    return idx, cnt


def second_order_spread(q, k, kbar, scale: float, *, with_rank=False, status=None, stream=None):
    """Gated second-order spread w [heads, nb, nb] with the pooled squared
    queries qsq and key variances kvar [heads, nb, d]: (w, qsq, kvar), plus
    the ranking bonus min(w, ln n_j) when ``with_rank``."""
    q, k, _ = _qkv(q, k, k)
    H, n, d = q.shape
    nb = -(-n // BLOCK)
    f = dict(device=q.device, dtype=torch.float32)
    qsq, kvar = torch.empty(H, nb, d, **f), torch.empty(H, nb, d, **f)
    w = torch.empty(H, nb, nb, **f)
    wrank = torch.empty(H, nb, nb, **f) if with_rank else None
    rc = load().pisa_second_order_spread(_ptr(q), _ptr(k), _dtype_code(q.dtype), H, n, d, BLOCK,
                                         float(scale), _ptr(kbar.contiguous()), _ptr(qsq),
                                         _ptr(kvar), _ptr(w), _ptr(wrank), _ptr(status),
                                         _stream(stream))
    _check(rc, "pisa_second_order_spread")
    return (w, qsq, kvar, wrank) if with_rank else (w, qsq, kvar)


def forward_second_order(q, k, v, idx, cnt, w, scale: float, *, out=None, out_dtype=None,
                         status=None, stream=None):
    """Piecewise output with the second-order block mass (spread w)."""
    q, k, v = _qkv(q, k, v)
    H, n, d = q.shape
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty(H, n, d, device=q.device, dtype=out_dtype)
    else:
        _check_out(out, (H, n, d), q.device)
    idx, cnt = idx.contiguous(), cnt.contiguous()
    rc = load().pisa_forward_second_order(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n,
                                          d, BLOCK, float(scale), _ptr(idx), _ptr(cnt),
                                          idx.shape[-1], _ptr(w.contiguous()), _ptr(out),
                                          _dtype_code(out.dtype), _ptr(status), _stream(stream))
    _check(rc, "pisa_forward_second_order")
    return out


def route_ex(qbar, kbar, scale: float, topk: int, band: int = 1, n_sink: int = 0, *,
             mnorm=None, eps: float = 1e-6, bonus=None, status=None, stream=None):
    """Critical block lists with the first ``n_sink`` key blocks forced in, the
    covariance-aware score when ``mnorm`` is given and a per-pair ``bonus``
    [heads, nb, nb] when given: idx, cnt."""
    qbar, kbar = qbar.contiguous(), kbar.contiguous()
    H, nb, d = qbar.shape
    ms = min(nb, topk + 2 * band + 1 + n_sink)
    idx = torch.empty(H, nb, ms, device=qbar.device, dtype=torch.int32)
    cnt = torch.empty(H, nb, device=qbar.device, dtype=torch.int32)
    rc = load().pisa_route_ex(_ptr(qbar), _ptr(kbar),
                              _ptr(mnorm.contiguous()) if mnorm is not None else None, float(eps),
                              _ptr(bonus.contiguous()) if bonus is not None else None, H, nb, d,
                              float(scale), int(topk), int(band), int(n_sink), _ptr(idx),
                              _ptr(cnt), ms, _ptr(status), _stream(stream))
    _check(rc, "pisa_route_ex")
    return idx, cnt


def morton_permutation(grid, n_prefix: int = 0, *, device=None, status=None, stream=None):
    """perm [n_prefix + T*Y*X] int32 (position -> source token) of the Morton order."""
    T, Y, X = grid
    device = device or torch.device("cuda")
    perm = torch.empty(n_prefix + T * Y * X, device=device, dtype=torch.int32)
    rc = load().pisa_morton_permutation(int(T), int(Y), int(X), int(n_prefix), _ptr(perm),
                                        _ptr(status), _stream(stream))
    _check(rc, "pisa_morton_permutation")
    return perm


def reorder_heads(x, perm, *, status=None, stream=None):
    """[n, heads, d] (token-major) -> [heads, n, d], row p of each head from token perm[p]."""
    x = x.contiguous()
    n, H, d = x.shape
    out = torch.empty(H, n, d, device=x.device, dtype=x.dtype)
    rc = load().pisa_reorder_heads(_ptr(x), _dtype_code(x.dtype), n, H, d, _ptr(perm.contiguous()),
                                   _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "pisa_reorder_heads")
    return out


def restore_heads(o, perm, *, status=None, stream=None):
    """Inverse of reorder_heads: [heads, n, d] -> [n, heads, d]."""
    o = o.contiguous()
    H, n, d = o.shape
    y = torch.empty(n, H, d, device=o.device, dtype=o.dtype)
    rc = load().pisa_restore_heads(_ptr(o), _dtype_code(o.dtype), n, H, d, _ptr(perm.contiguous()),
                                   _ptr(y), _ptr(status), _stream(stream))
    _check(rc, "pisa_restore_heads")
    return y


def forward(q, k, v, idx, cnt, scale: float, *, out=None, out_dtype=None, status=None,
            stream=None):
    """Piecewise attention output [heads, n, d]."""
    q, k, v = _qkv(q, k, v)
    H, n, d = q.shape
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty(H, n, d, device=q.device, dtype=out_dtype)
    else:
        _check_out(out, (H, n, d), q.device)
    idx, cnt = idx.contiguous(), cnt.contiguous()
    rc = load().pisa_forward(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n, d, BLOCK,
                             float(scale), _ptr(idx), _ptr(cnt), idx.shape[-1], _ptr(out),
                             _dtype_code(out.dtype), _ptr(status), _stream(stream))
    _check(rc, "pisa_forward")
    return out


def forward_hybrid(q, k, v, kbar, vsum, hbar, idx, cnt, scale: float, *, out=None,
                   out_dtype=None, workspace=None, status=None, stream=None):
    """Hybrid-order output [heads, n, d] (global first-order term). The bf16
    tensor-core path needs a scratch buffer; one is allocated here (torch's
    caching allocator) unless ``workspace`` (uint8, large enough) is given."""
    q, k, v = _qkv(q, k, v)
    H, n, d = q.shape
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty(H, n, d, device=q.device, dtype=out_dtype)
    else:
        _check_out(out, (H, n, d), q.device)
    idx, cnt = idx.contiguous(), cnt.contiguous()
    L = load()
    nbytes = L.pisa_forward_hybrid_workspace_size(_dtype_code(q.dtype), H, n, d)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = L.pisa_forward_hybrid(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n, d, BLOCK,
                               float(scale), _ptr(kbar.contiguous()), _ptr(vsum.contiguous()),
                               _ptr(hbar.contiguous()), _ptr(idx), _ptr(cnt), idx.shape[-1],
                               _ptr(out), _dtype_code(out.dtype), _ptr(workspace),
                               workspace.numel() if workspace is not None else 0, _ptr(status),
                               _stream(stream))
    _check(rc, "pisa_forward_hybrid")
    return out


def forward_hybrid_static(q, k, v, kbar, vsum, hbar, idx, cnt, scale: float, *, out,
                          status=None, stream=None):
    """pisa_forward_hybrid_static: the hybrid output written into the caller's
    ``out`` with no device allocation at all (library-owned fixed scratch;
    calls that overlap on the GPU must be serialised by the caller). Nothing
    is copied here either: every tensor must already have its exact shape,
    dtype and device and be contiguous, or ValueError / TypeError is raised."""
    if q.dim() != 3:
        raise ValueError("q must be [heads, n, d]")
    H, n, d = q.shape
    nb = -(-n // BLOCK)
    dev = q.device
    if not q.is_cuda or q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be a bfloat16 or float32 CUDA tensor")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(name, t, (H, n, d), q.dtype, dev)
    for name, t in (("kbar", kbar), ("vsum", vsum)):
        _require(name, t, (H, nb, d), torch.float32, dev)
    _require("hbar", hbar, (H, d, d), torch.float32, dev)
    if idx.dim() != 3:
        raise ValueError("idx must be [heads, nb, max_sel]")
    _require("idx", idx, (H, nb, idx.shape[-1]), torch.int32, dev)
    _require("cnt", cnt, (H, nb), torch.int32, dev)
    _check_out(out, (H, n, d), dev)
    if status is not None:
        _require("status", status, (1,), torch.int32, dev)
    rc = load().pisa_forward_hybrid_static(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n, d, BLOCK, float(scale),
        _ptr(kbar), _ptr(vsum), _ptr(hbar), _ptr(idx), _ptr(cnt), idx.shape[-1], _ptr(out),
        _dtype_code(out.dtype), _ptr(status), _stream(stream))
    _check(rc, "pisa_forward_hybrid_static")
    return out


def topk_for_density(density: float, nb: int) -> int:
    return int(math.ceil(density * nb - 1e-12))


def piecewise_sparse_attention(q, k, v, *, topk=None, density=None, band=1, scale=None,
                               variant="blockwise", routing="pooled", norm="spectral", eps=1e-6,
                               second_order=False, rank_bonus=False, n_sink=0, out=None,
                               out_dtype=None, status=None, stream=None):
    """Stats, route and forward on [heads, n, d] tensors. Give either ``topk``
    (blocks chosen besides the band) or ``density`` (topk = ceil(density nb)).

    variant:  "blockwise" (first-order term with each block's own H_j, Eq. 6)
              or "hybrid" (global Hbar, Eq. 10).
    routing:  "pooled" (s qbar.kbar) or "covariance" (plus log(M_j + eps),
              M_j = ||H_j - Hbar|| in ``norm``: Eq. 11).
    second_order: block-wise only; the gated second-order block mass
              n_j e^{a + w} of the Piecewise-Taylor-Attention README, and with
              ``rank_bonus`` its bounded bonus min(w, ln n_j) in the route.
    n_sink:   the first n_sink key blocks are exact for every query block.
    out:      optional output tensor [heads, n, d] (bf16 or float32)."""
    H, n, d = q.shape
    nb = -(-n // BLOCK)
    if variant not in ("blockwise", "hybrid"):
        raise ValueError(f"unknown variant {variant!r}")
    if routing not in ("pooled", "covariance"):
        raise ValueError(f"unknown routing {routing!r}")
    if second_order and variant != "blockwise":
        raise ValueError("second_order applies to the block-wise variant")
    if rank_bonus and not second_order:
        raise ValueError("rank_bonus needs second_order")
    if topk is None:
        topk = topk_for_density(0.125 if density is None else density, nb)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    kw = dict(status=status, stream=stream)
    need_hbar = variant == "hybrid" or routing == "covariance"
    qbar, kbar, vsum, _ = block_stats(q, k, v, with_vsum=need_hbar, **kw)
    hbar = global_first_order(k, v, kbar, vsum, **kw) if need_hbar else None
    mnorm = block_heterogeneity(k, v, kbar, hbar, norm=norm, **kw) if routing == "covariance" else None
    w = wrank = None
    if second_order:
        sp = second_order_spread(q, k, kbar, scale, with_rank=rank_bonus, **kw)
        w, wrank = sp[0], (sp[3] if rank_bonus else None)
    if mnorm is None and wrank is None and n_sink == 0:
        idx, cnt = route(qbar, kbar, scale, topk, band, **kw)
    else:
        idx, cnt = route_ex(qbar, kbar, scale, topk, band, n_sink, mnorm=mnorm, eps=eps,
                            bonus=wrank, **kw)
    if variant == "hybrid":
        return forward_hybrid(q, k, v, kbar, vsum, hbar, idx, cnt, scale, out=out,
                              out_dtype=out_dtype, **kw)
    if second_order:
        return forward_second_order(q, k, v, idx, cnt, w, scale, out=out, out_dtype=out_dtype, **kw)
    return forward(q, k, v, idx, cnt, scale, out=out, out_dtype=out_dtype, **kw)


def head_groups(heads: int, chunks: int, taper=False):
    """Bounds of ``chunks`` contiguous head groups. With ``taper`` the first
    and the last group get a smaller weight than the others (True: 1/2, or a
    float in (0, 1]): the upload of the first group and the download of the
    last one are the pipeline's exposed copies, so keeping them small
    shortens the whole."""
    chunks = max(1, min(int(chunks), heads))
    wts = [1.0] * chunks
    end = 0.5 if taper is True else float(taper or 1.0)
    if not 0.0 < end <= 1.0:
        raise ValueError("taper weight must be in (0, 1]")
    if chunks >= 3:
        wts[0] = wts[-1] = end
    tot, acc, bounds = sum(wts), 0.0, [0]
    for w in wts[:-1]:
        acc += w
        bounds.append(min(heads - (chunks - len(bounds)), max(bounds[-1] + 1, round(acc * heads / tot))))
    bounds.append(heads)
    return bounds


def piecewise_sparse_attention_host(q, k, v, out, *, topk=None, density=None, band=1, scale=None,
                                    chunks=4, taper=False, device=None, status=None, **options):
    """piecewise_sparse_attention on pinned HOST tensors [heads, n, d] (bf16 or
    f32), writing the pinned host ``out``; ``options`` are that function's
    (variant, routing, norm, eps, second_order, rank_bonus, n_sink). Heads are independent, so they go through
    in ``chunks`` groups (``taper``: smaller first and last groups, see
    head_groups): an upload stream moves group c + 1 to the device and
    a download stream moves group c - 1's output back while a compute stream
    runs stats, route and forward on group c (two compute streams alternate,
    so one group's last CTAs overlap the next group's launch). Device buffers
    are two groups deep. Returns after everything is enqueued on the current
    stream's timeline; synchronise before reading ``out``."""
    H, n, d = q.shape
    device = device or torch.device("cuda")
    nb = -(-n // BLOCK)
    if topk is None:
        topk = topk_for_density(0.125 if density is None else density, nb)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    bounds = head_groups(H, chunks, taper)
    chunks = len(bounds) - 1
    width = max(bounds[c + 1] - bounds[c] for c in range(chunks))
    with _host_lock:
        return _host_pipeline(q, k, v, out, bounds, width, device, topk, band, scale, status,
                              options)


def _host_pipeline(q, k, v, out, bounds, width, device, topk, band, scale, status, options):
    """The body of piecewise_sparse_attention_host, under _host_lock. Every
    call's streams first wait for the end of the previous call: its device
    buffers are shared, whichever thread or current stream made the call."""
    H, n, d = q.shape
    chunks = len(bounds) - 1
    key = (device, q.dtype, out.dtype, width, n, d)
    global _host_state
    prev_end = _host_state["end"] if _host_state is not None else None
    if _host_state is None or _host_state["key"] != key:
        mk = lambda dt: [torch.empty(width, n, d, device=device, dtype=dt) for _ in range(2)]
        _host_state = {
            "key": key, "q": mk(q.dtype), "k": mk(q.dtype), "v": mk(q.dtype), "o": mk(out.dtype),
            "up": torch.cuda.Stream(device), "down": torch.cuda.Stream(device),
            "comp": [torch.cuda.Stream(device) for _ in range(2)], "end": None,
        }
    S = _host_state
    cur = torch.cuda.current_stream(device)
    up, down = S["up"], S["down"]
    consumed = [None, None]  # compute done with buffer b (inputs read, output written)
    drained = [None, None]   # output of buffer b copied back
    for st in (up, down, *S["comp"]):
        st.wait_stream(cur)
        if prev_end is not None:
            st.wait_event(prev_end)
    for c in range(chunks):
        h0, h1 = bounds[c], bounds[c + 1]
        w = h1 - h0
        b = c % 2
        with torch.cuda.stream(up):
            if consumed[b] is not None:
                up.wait_event(consumed[b])
            for src, dst in ((q, S["q"][b]), (k, S["k"][b]), (v, S["v"][b])):
                dst[:w].copy_(src[h0:h1], non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up)
        comp = S["comp"][b]
        comp.wait_event(loaded)
        if drained[b] is not None:
            comp.wait_event(drained[b])
        dq, dk, dv, do = S["q"][b][:w], S["k"][b][:w], S["v"][b][:w], S["o"][b][:w]
        with torch.cuda.stream(comp):
            piecewise_sparse_attention(dq, dk, dv, topk=topk, band=band, scale=scale, out=do,
                                       status=status, stream=comp, **options)
        consumed[b] = torch.cuda.Event()
        consumed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(consumed[b])
            out[h0:h1].copy_(do, non_blocking=True)
            drained[b] = torch.cuda.Event()
            drained[b].record(down)
    for st in (up, down, *S["comp"]):
        cur.wait_stream(st)
    S["end"] = torch.cuda.Event()
    S["end"].record(cur)
    return out


_host_state = None
_host_lock = threading.Lock()


def attention_host_workspace(q, out, topk, band, groups, taper, device=None):
    """A device workspace (uint8) large enough for attention_host."""
    H, n, d = q.shape
    nbytes = load().pisa_attention_host_workspace_size(_dtype_code(q.dtype), _dtype_code(out.dtype),
                                                       H, n, d, int(topk), int(band), int(groups),
                                                       int(bool(taper)))
    return torch.empty(nbytes + 256, device=device or "cuda", dtype=torch.uint8)


def attention_host(q, k, v, out, *, topk, band=1, scale=None, groups=10, taper=True,
                   workspace=None, status=None, stream=None):
    """pisa_attention_host: stats, route and block-wise forward on pinned HOST
    tensors q, k, v [heads, n, d] into the pinned HOST tensor ``out``, in C
    (copies, streams and events included). Returns after enqueuing on
    ``stream`` (the current stream by default); synchronise before reading
    ``out``. ``workspace``: a device uint8 tensor from
    attention_host_workspace (allocated here when None)."""
    if q.dim() != 3 or q.shape != k.shape or q.shape != v.shape or out.shape != q.shape:
        raise ValueError("q, k, v and out must share the shape [heads, n, d]")
    if q.is_cuda or k.is_cuda or v.is_cuda or out.is_cuda:
        raise ValueError("attention_host takes host tensors")
    for t in (q, k, v, out):
        if not t.is_contiguous():
            raise ValueError("host tensors must be contiguous")
    H, n, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if workspace is None:
        workspace = attention_host_workspace(q, out, topk, band, groups, taper)
    base = workspace.data_ptr()
    off = (-base) % 256  # the call wants a 256-byte aligned workspace
    rc = load().pisa_attention_host(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), H, n, d, BLOCK,
                                    float(scale), int(topk), int(band), _ptr(out),
                                    _dtype_code(out.dtype), int(groups), int(bool(taper)),
                                    ctypes.c_void_p(base + off), workspace.numel() - off,
                                    _ptr(status), _stream(stream))
    _check(rc, "pisa_attention_host")
    return out


def selftest_tc(a, b, bt, mode: int = 0, *, status=None, stream=None):
    """Diagnostic tensor-core product (see include/pisa_selftest.h)."""
    out = torch.zeros(4, 128, 128, device=a.device, dtype=torch.float32)
    rc = load().pisa_selftest_tc(_ptr(a.contiguous()), _ptr(b.contiguous()),
                                 _ptr(bt.contiguous()), _ptr(out), int(mode), _ptr(status),
                                 _stream(stream))
    _check(rc, "pisa_selftest_tc")
    return out
