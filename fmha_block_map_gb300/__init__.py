"""LUT-driven block-sparse attention forward on GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libfbm.so`` (``include/fbm.h``).
Every function here only marshals arguments: it takes torch tensors, checks
their dtype / device / contiguity, allocates outputs with torch when the caller
passes none, and calls the C entry point of the same name on the current CUDA
stream.  All computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback.  If the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence, Union

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfbm.so")

FBM_OK, FBM_ERR_INVALID_ARG, FBM_ERR_UNSUPPORTED, FBM_ERR_CUDA, FBM_ERR_DEVICE = range(5)
FBM_F16, FBM_BF16, FBM_F32 = 0, 1, 2
FBM_DEVERR_LUT_RANGE, FBM_DEVERR_TIMEOUT, FBM_DEVERR_LUT_ORDER = 0x1, 0x2, 0x4
FBM_MAX_HEADS = 256
FBM_STATIC_SCRATCH_BYTES = 32 << 20

_lib = None


class FbmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libfbm status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run fmha_block_map_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        L.fbm_version.restype = i32
        L.fbm_last_error_message.restype = ctypes.c_char_p
        L.fbm_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.fbm_block_map_workspace_bytes.argtypes = [i32] * 7
        L.fbm_block_map_workspace_bytes.restype = sz
        L.sparge_block_map.argtypes = ([vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                        f32, i32, i32, i32, vp, vp, vp, vp, sz, vp])
        L.sparge_block_map_static.argtypes = ([vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp,
                                               vp, f32, i32, i32, i32, vp, vp, vp, vp])
        L.sparge_block_map_e4m3.argtypes = ([vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp,
                                             vp, f32, i32, i32, i32, vp, vp, vp, vp, sz, vp, vp, vp,
                                             vp, vp])
        L.sparse_fmha_fwd.argtypes = ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                       vp, vp, i32, i32, f32, i32, i32, f32, vp, vp, vp, vp, vp])
        L.attn_combine.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, vp]
        L.lut_shard.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, i32, vp]
        L.lut_validate.argtypes = [vp, vp, i64, i32, i32, vp]
        L.lut_pair_union.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, i32, vp]
        L.sparse_fmha_fwd_pairs.argtypes = ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                             vp, vp, i32, f32, i32, i32, vp, vp, vp])
        L.quantize_e4m3_blocks.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp]
        L.sparse_fmha_fwd_fp8.argtypes = ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                           i32, vp, vp, i32, f32, i32, vp, vp, vp])
        L.sparse_decode_fwd.argtypes = ([vp, vp, i32, i32, i32, i32, i32, i32, i64, vp, i32, vp,
                                         i32, i32, f32, vp, vp, vp])
        L.fbm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.fbm_selftest_wait_timeout.restype = i32
        L.fbm_fmha_kernel_kind.argtypes = [i32] * 6
        L.fbm_fmha_kernel_kind.restype = i32
        for name in ("fbm_get_error", "sparge_block_map", "sparge_block_map_static",
                     "sparse_fmha_fwd", "attn_combine", "lut_shard", "lut_validate",
                     "lut_pair_union", "sparse_fmha_fwd_pairs",
                     "sparse_decode_fwd",
                     "quantize_e4m3_blocks", "sparse_fmha_fwd_fp8"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != FBM_OK:
        raise FbmError(status, lib().fbm_last_error_message().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FBM_F16
    if t.dtype == torch.bfloat16:
        return FBM_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _per_head(x, hq: int, name: str):
    if x is None:
        return None
    if isinstance(x, (int, float)):
        arr = (ctypes.c_float * hq)(*([float(x)] * hq))
    else:
        vals = [float(v) for v in x]
        if len(vals) != hq:
            raise ValueError(f"{name} needs {hq} values")
        arr = (ctypes.c_float * hq)(*vals)
    return arr


def version() -> int:
    return lib().fbm_version()


def get_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits."""
    detail = ctypes.c_uint32(0)
    st = lib().fbm_get_error(_stream(stream), ctypes.byref(detail))
    if st not in (FBM_OK, FBM_ERR_DEVICE):
        _check(st)
    return int(detail.value)


def block_map_workspace_bytes(b: int, hq: int, hk: int, s: int, d: int) -> int:
    return int(lib().fbm_block_map_workspace_bytes(b, hq, hk, s, d, 64, 64))


def sparge_block_map(q: torch.Tensor, k: torch.Tensor, *, topk=None, cdfthreshd=None,
                     simthreshd1: Union[float, Sequence[float]] = 0.001,
                     scale: Optional[float] = None, causal: bool = False,
                     attention_sink: bool = False, return_block_map: bool = False,
                     lut: Optional[torch.Tensor] = None, lut_count: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, smooth_k: bool = False,
                     stream=None):
    """Block map of q [b, hq, s, d] against k [b, hk, s, d]; returns
    (lut [b, hq, nq, nk] int32, lut_count [b, hq, nq] int32, block_map or None).
    topk / cdfthreshd / simthreshd1 are a float or one value per query head;
    smooth_k subtracts the mean key row of each (batch, KV head) first."""
    _cuda(q, "q"), _cuda(k, "k")
    b, hq, s, d = q.shape
    hk = k.shape[1]
    nq = (s + 63) // 64
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if lut is None:
        lut = torch.empty((b, hq, nq, nq), dtype=torch.int32, device=dev)
    if lut_count is None:
        lut_count = torch.empty((b, hq, nq), dtype=torch.int32, device=dev)
    bmap = torch.empty((b, hq, nq, nq), dtype=torch.uint8, device=dev) if return_block_map else None
    need = block_map_workspace_bytes(b, hq, hk, s, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(lib().sparge_block_map(
        _ptr(q), _ptr(k), _dt(q), b, hq, hk, s, d, 64, 64,
        _per_head(topk, hq, "topk"), _per_head(cdfthreshd, hq, "cdfthreshd"),
        _per_head(simthreshd1, hq, "simthreshd1"), float(scale), int(causal),
        int(attention_sink), int(smooth_k), _ptr(lut), _ptr(lut_count), _ptr(bmap),
        _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return lut, lut_count, bmap


def sparge_block_map_e4m3(q: torch.Tensor, k: torch.Tensor, *, topk=None, cdfthreshd=None,
                          simthreshd1: Union[float, Sequence[float]] = 0.001,
                          scale: Optional[float] = None, causal: bool = False,
                          attention_sink: bool = False, return_block_map: bool = False,
                          lut: Optional[torch.Tensor] = None,
                          lut_count: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, smooth_k: bool = False,
                          q8: Optional[torch.Tensor] = None, q_scale: Optional[torch.Tensor] = None,
                          k8: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
                          stream=None):
    """sparge_block_map plus the e4m3 codes and per-block scales of q and k
    (those of quantize_e4m3_blocks) from the same pass; d = 128.  Returns
    (lut, lut_count, block_map or None, q8, q_scale, k8, k_scale)."""
    _cuda(q, "q"), _cuda(k, "k")
    b, hq, s, d = q.shape
    hk = k.shape[1]
    nq = (s + 63) // 64
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if lut is None:
        lut = torch.empty((b, hq, nq, nq), dtype=torch.int32, device=dev)
    if lut_count is None:
        lut_count = torch.empty((b, hq, nq), dtype=torch.int32, device=dev)
    bmap = torch.empty((b, hq, nq, nq), dtype=torch.uint8, device=dev) if return_block_map else None
    need = block_map_workspace_bytes(b, hq, hk, s, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if q8 is None:
        q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    if k8 is None:
        k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    if q_scale is None:
        q_scale = torch.empty((b, hq, nq), dtype=torch.float32, device=dev)
    if k_scale is None:
        k_scale = torch.empty((b, hk, nq), dtype=torch.float32, device=dev)
    _check(lib().sparge_block_map_e4m3(
        _ptr(q), _ptr(k), _dt(q), b, hq, hk, s, d, 64, 64,
        _per_head(topk, hq, "topk"), _per_head(cdfthreshd, hq, "cdfthreshd"),
        _per_head(simthreshd1, hq, "simthreshd1"), float(scale), int(causal),
        int(attention_sink), int(smooth_k), _ptr(lut), _ptr(lut_count), _ptr(bmap),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(q8), _ptr(q_scale),
        _ptr(k8), _ptr(k_scale), _stream(stream)))
    return lut, lut_count, bmap, q8, q_scale, k8, k_scale


def sparge_block_map_static(q: torch.Tensor, k: torch.Tensor, *, topk=None, cdfthreshd=None,
                            simthreshd1: Union[float, Sequence[float]] = 0.001,
                            scale: Optional[float] = None, causal: bool = False,
                            attention_sink: bool = False, return_block_map: bool = False,
                            lut: Optional[torch.Tensor] = None,
                            lut_count: Optional[torch.Tensor] = None, smooth_k: bool = False,
                            stream=None):
    """sparge_block_map with the library's static scratch array instead of a
    workspace, for callers that cannot allocate device scratch (the outputs
    are still the caller's: pass lut / lut_count to allocate nothing here)."""
    _cuda(q, "q"), _cuda(k, "k")
    b, hq, s, d = q.shape
    hk = k.shape[1]
    nq = (s + 63) // 64
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if lut is None:
        lut = torch.empty((b, hq, nq, nq), dtype=torch.int32, device=dev)
    if lut_count is None:
        lut_count = torch.empty((b, hq, nq), dtype=torch.int32, device=dev)
    bmap = torch.empty((b, hq, nq, nq), dtype=torch.uint8, device=dev) if return_block_map else None
    _check(lib().sparge_block_map_static(
        _ptr(q), _ptr(k), _dt(q), b, hq, hk, s, d, 64, 64,
        _per_head(topk, hq, "topk"), _per_head(cdfthreshd, hq, "cdfthreshd"),
        _per_head(simthreshd1, hq, "simthreshd1"), float(scale), int(causal),
        int(attention_sink), int(smooth_k), _ptr(lut), _ptr(lut_count), _ptr(bmap),
        _stream(stream)))
    return lut, lut_count, bmap


def sparse_fmha_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    lut: Optional[torch.Tensor], lut_count: Optional[torch.Tensor], *,
                    scale: Optional[float] = None, causal: bool = False, key_offset: int = 0,
                    return_lse: bool = False, num_splits: int = 1,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    o_partial: Optional[torch.Tensor] = None,
                    lse_partial: Optional[torch.Tensor] = None, partial: bool = False,
                    pv_threshold: Optional[float] = None, stream=None):
    """Sparse (lut given) or dense (lut None) attention.  num_splits == 1
    returns (out, lse or None); num_splits > 1, or ``partial`` (one whole-row
    partial, e.g. one slot of a context-parallel stack), returns the fp32
    partials (o_partial [S, b, hq, s_q, dv], lse_partial [S, b, hq, s_q]).
    pv_threshold (None: off) enables the per-Q-tile PV skip on whole rows.
    Under causal, key index u is visible to query row t when
    u <= t + key_offset (0: queries and keys start at the same position)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _cuda(t, n)
    b, hq, s_q, d = q.shape
    hk, s_k, dv = k.shape[1], k.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    stride = 0
    if lut is not None:
        _cuda(lut, "lut"), _cuda(lut_count, "lut_count")
        if lut.dtype != torch.int32 or lut_count.dtype != torch.int32:
            raise TypeError("lut / lut_count must be int32")
        stride = lut.shape[-1]
    dev = q.device
    partial = partial or num_splits > 1
    if not partial:
        if out is None:
            out = torch.empty((b, hq, s_q, dv), dtype=q.dtype, device=dev)
        if return_lse and lse is None:
            lse = torch.empty((b, hq, s_q), dtype=torch.float32, device=dev)
    else:
        if o_partial is None:
            o_partial = torch.empty((num_splits, b, hq, s_q, dv), dtype=torch.float32, device=dev)
        if lse_partial is None:
            lse_partial = torch.empty((num_splits, b, hq, s_q), dtype=torch.float32, device=dev)
    _check(lib().sparse_fmha_fwd(
        _ptr(q), _ptr(k), _ptr(v), _dt(q), b, hq, hk, s_q, s_k, d, dv, 64, 64,
        _ptr(lut), _ptr(lut_count), stride, num_splits, float(scale), int(causal), int(key_offset),
        math.inf if pv_threshold is None else float(pv_threshold),
        None if partial else _ptr(out), None if partial else _ptr(lse),
        _ptr(o_partial) if partial else None, _ptr(lse_partial) if partial else None,
        _stream(stream)))
    if not partial:
        return out, lse
    return o_partial, lse_partial


def attn_combine(o_part: torch.Tensor, lse_part: torch.Tensor, *, out_dtype=torch.float32,
                 out: Optional[torch.Tensor] = None, return_lse: bool = True, stream=None):
    """Merge partials o_part [S, ..., dv] (fp32) / lse_part [S, ...] into
    (out [..., dv], lse [...] or None)."""
    _cuda(o_part, "o_part"), _cuda(lse_part, "lse_part")
    S = o_part.shape[0]
    dv = o_part.shape[-1]
    rows = lse_part[0].numel()
    codes = {torch.float16: FBM_F16, torch.bfloat16: FBM_BF16, torch.float32: FBM_F32}
    if out is None:
        out = torch.empty(o_part.shape[1:], dtype=out_dtype, device=o_part.device)
    lse = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=o_part.device) \
        if return_lse else None
    _check(lib().attn_combine(_ptr(o_part), _ptr(lse_part), S, rows, dv, codes[out.dtype],
                              _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def quantize_e4m3_blocks(x: torch.Tensor, *, codes: Optional[torch.Tensor] = None,
                         scales: Optional[torch.Tensor] = None, stream=None):
    """x [..., s, 128] fp16 / bf16 -> (codes uint8 [..., s, 128], scales fp32
    [..., ceil(s / 64)]): e4m3 codes with one scale per 64-row block."""
    _cuda(x, "x")
    s, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    bh = 1
    for n in lead:
        bh *= n
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(lead + ((s + 63) // 64,), dtype=torch.float32, device=x.device)
    _check(lib().quantize_e4m3_blocks(_ptr(x), _dt(x), bh, s, d, _ptr(codes), _ptr(scales),
                                      _stream(stream)))
    return codes, scales


def sparse_fmha_fwd_fp8(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor,
                        k_scale: torch.Tensor, v: torch.Tensor, lut: Optional[torch.Tensor],
                        lut_count: Optional[torch.Tensor], *, scale: Optional[float] = None,
                        causal: bool = False, return_lse: bool = False,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        stream=None):
    """Sparse attention with e4m3 Q / K (from quantize_e4m3_blocks) and
    16-bit V: returns (out [b, hq, s_q, 128] in v's dtype, lse or None)."""
    for t_, n in ((q8, "q8"), (q_scale, "q_scale"), (k8, "k8"), (k_scale, "k_scale"), (v, "v")):
        _cuda(t_, n)
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8:
        raise TypeError("q8 / k8 must be uint8 e4m3 codes")
    b, hq, s_q, d = q8.shape
    hk, s_k, dv = k8.shape[1], k8.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    stride = 0
    if lut is not None:
        _cuda(lut, "lut"), _cuda(lut_count, "lut_count")
        if lut.dtype != torch.int32 or lut_count.dtype != torch.int32:
            raise TypeError("lut / lut_count must be int32")
        stride = lut.shape[-1]
    if out is None:
        out = torch.empty((b, hq, s_q, dv), dtype=v.dtype, device=v.device)
    if return_lse and lse is None:
        lse = torch.empty((b, hq, s_q), dtype=torch.float32, device=v.device)
    _check(lib().sparse_fmha_fwd_fp8(
        _ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(v), _dt(v), b, hq, hk, s_q, s_k,
        d, dv, _ptr(lut), _ptr(lut_count), stride, float(scale), int(causal), _ptr(out),
        _ptr(lse), _stream(stream)))
    return out, lse


def lut_shard(lut: torch.Tensor, lut_count: torch.Tensor, lo: int, hi: int, *,
              out_lut: Optional[torch.Tensor] = None, out_count: Optional[torch.Tensor] = None,
              stream=None):
    """The entries of every LUT row (lut [..., stride], lut_count [...]) inside
    the kv-block range [lo, hi), re-based to lo: (out_lut [..., hi - lo],
    out_count [...]), -1 padded."""
    _cuda(lut, "lut"), _cuda(lut_count, "lut_count")
    if lut.dtype != torch.int32 or lut_count.dtype != torch.int32:
        raise TypeError("lut / lut_count must be int32")
    lead = tuple(lut.shape[:-1])
    if tuple(lut_count.shape) != lead:
        raise ValueError("lut_count must have the shape of lut without its last dimension")
    if out_lut is None:
        out_lut = torch.empty(lead + (hi - lo,), dtype=torch.int32, device=lut.device)
    if out_count is None:
        out_count = torch.empty(lead, dtype=torch.int32, device=lut.device)
    _cuda(out_lut, "out_lut"), _cuda(out_count, "out_count")
    if tuple(out_lut.shape[:-1]) != lead or tuple(out_count.shape) != lead:
        raise ValueError("out_lut / out_count must have the leading shape of lut")
    _check(lib().lut_shard(_ptr(lut), _ptr(lut_count), lut_count.numel(), lut.shape[-1], lo, hi,
                           _ptr(out_lut), _ptr(out_count), out_lut.shape[-1], _stream(stream)))
    return out_lut, out_count


def lut_validate(lut: torch.Tensor, lut_count: torch.Tensor, nk: int, *, stream=None) -> int:
    """Check lut [..., stride] / lut_count [...] (int32) against the contract of
    sparse_fmha_fwd: counts in [0, min(nk, stride)], entries in [0, nk),
    strictly ascending.  Returns the device error bits found
    (FBM_DEVERR_LUT_RANGE | FBM_DEVERR_LUT_ORDER; 0: valid); synchronises."""
    _cuda(lut, "lut"), _cuda(lut_count, "lut_count")
    if lut.dtype != torch.int32 or lut_count.dtype != torch.int32:
        raise TypeError("lut / lut_count must be int32")
    if tuple(lut_count.shape) != tuple(lut.shape[:-1]):
        raise ValueError("lut_count must have the shape of lut without its last dimension")
    _check(lib().lut_validate(_ptr(lut), _ptr(lut_count), lut_count.numel(), lut.shape[-1], nk,
                              _stream(stream)))
    return get_error(stream)


def lut_pair_union(lut: torch.Tensor, lut_count: torch.Tensor, nk: int, *,
                   pair_lut: Optional[torch.Tensor] = None,
                   pair_count: Optional[torch.Tensor] = None, stream=None):
    """lut [b, hq, nq, stride] / lut_count [b, hq, nq] -> (pair_lut [b, hq,
    ceil(nq / 2), nk], pair_count [b, hq, ceil(nq / 2)]): the union of the
    LUT rows of q blocks 2p and 2p + 1, ascending, each entry
    j | (in row 2p) << 29 | (in row 2p + 1) << 30."""
    _cuda(lut, "lut"), _cuda(lut_count, "lut_count")
    if lut.dtype != torch.int32 or lut_count.dtype != torch.int32:
        raise TypeError("lut / lut_count must be int32")
    *lead, nq, stride = lut.shape
    bh = 1
    for n in lead:
        bh *= n
    npq = (nq + 1) // 2
    if pair_lut is None:
        pair_lut = torch.empty(tuple(lead) + (npq, nk), dtype=torch.int32, device=lut.device)
    if pair_count is None:
        pair_count = torch.empty(tuple(lead) + (npq,), dtype=torch.int32, device=lut.device)
    _check(lib().lut_pair_union(_ptr(lut), _ptr(lut_count), bh, nq, stride, nk, _ptr(pair_lut),
                                _ptr(pair_count), pair_lut.shape[-1], _stream(stream)))
    return pair_lut, pair_count


def sparse_fmha_fwd_pairs(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          pair_lut: Optional[torch.Tensor], pair_count: Optional[torch.Tensor], *,
                          scale: Optional[float] = None, causal: bool = False,
                          key_offset: int = 0, return_lse: bool = False,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          stream=None):
    """sparse_fmha_fwd (whole rows) on 128-row tiles of q-block pairs:
    pair_lut / pair_count from lut_pair_union (None: dense).  Returns
    (out, lse or None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _cuda(t, n)
    b, hq, s_q, d = q.shape
    hk, s_k, dv = k.shape[1], k.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    stride = 0
    if pair_lut is not None:
        _cuda(pair_lut, "pair_lut"), _cuda(pair_count, "pair_count")
        if pair_lut.dtype != torch.int32 or pair_count.dtype != torch.int32:
            raise TypeError("pair_lut / pair_count must be int32")
        stride = pair_lut.shape[-1]
    if out is None:
        out = torch.empty((b, hq, s_q, dv), dtype=q.dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((b, hq, s_q), dtype=torch.float32, device=q.device)
    _check(lib().sparse_fmha_fwd_pairs(
        _ptr(q), _ptr(k), _ptr(v), _dt(q), b, hq, hk, s_q, s_k, d, dv, _ptr(pair_lut),
        _ptr(pair_count), stride, float(scale), int(causal), int(key_offset), _ptr(out),
        _ptr(lse), _stream(stream)))
    return out, lse


def sparse_decode_fwd(q: torch.Tensor, kv_cache: torch.Tensor, page_table: torch.Tensor,
                      indices: torch.Tensor, *, dv: int, scale: float, num_splits: int = 1,
                      o_partial: Optional[torch.Tensor] = None,
                      lse_partial: Optional[torch.Tensor] = None, stream=None):
    """Split-KV partials of sparse decode: q [n_q, hq, d], kv_cache
    [n_pages, page, d], page_table [n_q, pages_per_query] int32, indices
    [n_q, topk] int32.  Returns (o_partial [S, n_q, hq, dv], lse_partial
    [S, n_q, hq]) in fp32."""
    for t, n in ((q, "q"), (kv_cache, "kv_cache"), (page_table, "page_table"),
                 (indices, "indices")):
        _cuda(t, n)
    n_q, hq, d = q.shape
    n_pages, page, _ = kv_cache.shape
    dev = q.device
    if o_partial is None:
        o_partial = torch.empty((num_splits, n_q, hq, dv), dtype=torch.float32, device=dev)
    if lse_partial is None:
        lse_partial = torch.empty((num_splits, n_q, hq), dtype=torch.float32, device=dev)
    _check(lib().sparse_decode_fwd(
        _ptr(q), _ptr(kv_cache), _dt(q), n_q, hq, d, dv, page, n_pages, _ptr(page_table),
        page_table.shape[1], _ptr(indices), indices.shape[1], num_splits, float(scale),
        _ptr(o_partial), _ptr(lse_partial), _stream(stream)))
    return o_partial, lse_partial


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Run the bounded-wait expiry path on the GPU (see include/fbm.h)."""
    _check(lib().fbm_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def fmha_kernel_kind(dtype: torch.dtype, d: int, dv: int, num_splits: int, s_q: int,
                     s_k: int) -> int:
    """1 = the tcgen05 kernel, 0 = rejected."""
    code = {torch.float16: FBM_F16, torch.bfloat16: FBM_BF16}[dtype]
    return int(lib().fbm_fmha_kernel_kind(code, d, dv, num_splits, s_q, s_k))
