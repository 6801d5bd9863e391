"""The C ABI library loads, exports every entry point include/fbm.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import fmha_block_map_gb300 as fbm
from fmha_block_map_gb300 import build as fbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fbm.h")


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fbm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) -
                  {"defined", "sizeof", "extern"})


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sparge_block_map", "sparse_fmha_fwd", "attn_combine", "sparse_decode_fwd",
              "fbm_get_error", "fbm_block_map_workspace_bytes", "fbm_last_error_message",
              "fbm_version", "fbm_fmha_kernel_kind"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"libfbm.so does not export {n}"
    assert L.fbm_version() == 100


def test_workspace_size(L):
    n = fbm.block_map_workspace_bytes(2, 32, 32, 16384, 128)
    # pooled means (fp32) and sims (fp32) of 2*32*256 q and k blocks, the mean key rows of
    # 2*32 KV heads, 256-B aligned pieces
    assert n >= 2 * (2 * 32 * 256 * 128 * 4 + 2 * 32 * 256 * 4) + 2 * 32 * 128 * 4
    assert L.fbm_block_map_workspace_bytes(1, 1, 1, 64, 64, 32, 64) == 0
    L.fbm_workspace_bytes.restype = ctypes.c_size_t
    assert L.fbm_workspace_bytes(2, 32, 32, 16384, 128) == n


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: checks fail before any launch


def _bm(L, **kw):
    a = dict(q=FAKE, k=FAKE, dtype=0, b=1, hq=2, hk=2, s=512, d=64, blkq=64, blkk=64,
             topk=(ctypes.c_float * 2)(0.5, 0.5), cdf=None,
             sim=(ctypes.c_float * 2)(0.001, 0.001), scale=0.125, causal=0, sink=0, smooth=0,
             lut=FAKE, cnt=FAKE, bmap=None, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return L.sparge_block_map(a["q"], a["k"], a["dtype"], a["b"], a["hq"], a["hk"], a["s"],
                              a["d"], a["blkq"], a["blkk"], a["topk"], a["cdf"], a["sim"],
                              a["scale"], a["causal"], a["sink"], a["smooth"], a["lut"], a["cnt"],
                              a["bmap"],
                              a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fbm.FBM_ERR_INVALID_ARG),
    (dict(hq=3, topk=(ctypes.c_float * 3)(.5, .5, .5), sim=(ctypes.c_float * 3)(0, 0, 0)),
     fbm.FBM_ERR_INVALID_ARG),
    (dict(d=96), fbm.FBM_ERR_UNSUPPORTED),
    (dict(blkq=128), fbm.FBM_ERR_UNSUPPORTED),
    (dict(cdf=(ctypes.c_float * 2)(0.9, 0.9)), fbm.FBM_ERR_INVALID_ARG),  # both modes
    (dict(topk=None), fbm.FBM_ERR_INVALID_ARG),                            # neither
    (dict(topk=(ctypes.c_float * 2)(0.0, 0.5)), fbm.FBM_ERR_INVALID_ARG),
    (dict(topk=(ctypes.c_float * 2)(1.5, 0.5)), fbm.FBM_ERR_INVALID_ARG),
    (dict(wsb=16), fbm.FBM_ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p((1 << 20) + 4)), fbm.FBM_ERR_INVALID_ARG),
    (dict(dtype=7), fbm.FBM_ERR_INVALID_ARG),
    (dict(s=70000), fbm.FBM_ERR_UNSUPPORTED),
    (dict(scale=0.0), fbm.FBM_ERR_INVALID_ARG),
])
def test_block_map_rejects(L, kw, code):
    assert _bm(L, **kw) == code
    assert L.fbm_last_error_message()


def _fm(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, b=1, hq=4, hk=2, s_q=256, s_k=256, d=128, dv=128,
             blkq=64, blkk=64, lut=FAKE, cnt=FAKE, stride=4, S=1, scale=0.1, causal=0, koff=0,
             pv=float("inf"), out=FAKE, lse=None, op=None, lp=None)
    a.update(kw)
    return L.sparse_fmha_fwd(a["q"], a["k"], a["v"], a["dtype"], a["b"], a["hq"], a["hk"],
                             a["s_q"], a["s_k"], a["d"], a["dv"], a["blkq"], a["blkk"],
                             a["lut"], a["cnt"], a["stride"], a["S"], a["scale"], a["causal"],
                             a["koff"], a["pv"], a["out"], a["lse"], a["op"], a["lp"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(v=None), fbm.FBM_ERR_INVALID_ARG),
    (dict(cnt=None), fbm.FBM_ERR_INVALID_ARG),
    (dict(hk=3), fbm.FBM_ERR_INVALID_ARG),
    (dict(d=96, dv=96), fbm.FBM_ERR_UNSUPPORTED),
    (dict(dv=64), fbm.FBM_ERR_UNSUPPORTED),
    (dict(causal=1, koff=(1 << 30) + 1), fbm.FBM_ERR_INVALID_ARG),
    (dict(S=2), fbm.FBM_ERR_INVALID_ARG),      # split without partial buffers
    (dict(S=0), fbm.FBM_ERR_INVALID_ARG),
    (dict(out=None), fbm.FBM_ERR_INVALID_ARG),
    (dict(stride=0), fbm.FBM_ERR_INVALID_ARG),
    (dict(blkk=128), fbm.FBM_ERR_UNSUPPORTED),
    (dict(k=ctypes.c_void_p((1 << 20) + 2)), fbm.FBM_ERR_INVALID_ARG),
    (dict(pv=float("nan")), fbm.FBM_ERR_INVALID_ARG),
    (dict(pv=-1.0), fbm.FBM_ERR_INVALID_ARG),
    (dict(pv=4.0, S=2, out=None, op=FAKE, lp=FAKE), fbm.FBM_ERR_UNSUPPORTED),   # split
    (dict(pv=4.0, out=None, op=FAKE, lp=FAKE), fbm.FBM_ERR_UNSUPPORTED),        # partial
])
def test_fmha_rejects(L, kw, code):
    assert _fm(L, **kw) == code


def test_combine_and_decode_reject(L):
    assert L.attn_combine(FAKE, FAKE, 0, 10, 128, 2, FAKE, None, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.attn_combine(FAKE, FAKE, 2, 10, 130, 2, FAKE, None, None) == fbm.FBM_ERR_UNSUPPORTED
    assert L.attn_combine(FAKE, None, 2, 10, 128, 2, FAKE, None, None) == fbm.FBM_ERR_INVALID_ARG
    args = [FAKE, FAKE, 1, 64, 16, 576, 512, 64, 65536, FAKE, 1024, FAKE, 2048, 4, 0.12,
            FAKE, FAKE, None]
    bad = list(args)
    bad[4] = 8  # hq
    assert L.sparse_decode_fwd(*bad) == fbm.FBM_ERR_UNSUPPORTED
    bad = list(args)
    bad[13] = 0  # splits
    assert L.sparse_decode_fwd(*bad) == fbm.FBM_ERR_INVALID_ARG
    bad = list(args)
    bad[9] = None  # page table
    assert L.sparse_decode_fwd(*bad) == fbm.FBM_ERR_INVALID_ARG


def test_lut_validate_rejects(L):
    assert L.lut_validate(None, FAKE, 4, 8, 8, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.lut_validate(FAKE, FAKE, 0, 8, 8, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.lut_validate(FAKE, FAKE, 4, 0, 8, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.lut_validate(FAKE, FAKE, 4, 8, 0, None) == fbm.FBM_ERR_INVALID_ARG


def test_lut_shard_rejects(L):
    # valid apart from the one bad argument each case plants; never called as is
    args = [FAKE, FAKE, 10, 16, 4, 8, FAKE, FAKE, 4, None]
    for i, bad in ((0, None), (2, 0), (3, 0), (4, -1), (5, 4), (8, 3)):
        a = list(args)
        a[i] = bad
        assert L.lut_shard(*a) == fbm.FBM_ERR_INVALID_ARG, (i, bad)


def test_fp8_entry_points_reject(L):
    q = [FAKE, 0, 2, 512, 128, FAKE, FAKE, None]
    for i, bad in ((0, None), (1, 7), (2, 0), (4, 64), (5, None)):
        a = list(q)
        a[i] = bad
        assert L.quantize_e4m3_blocks(*a) in (fbm.FBM_ERR_INVALID_ARG, fbm.FBM_ERR_UNSUPPORTED)
    f = [FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 4, 2, 256, 256, 128, 128, FAKE, FAKE, 4, 0.1, 0,
         FAKE, None, None]
    for i, bad, code in ((1, None, fbm.FBM_ERR_INVALID_ARG), (8, 3, fbm.FBM_ERR_INVALID_ARG),
                         (11, 64, fbm.FBM_ERR_UNSUPPORTED), (14, None, fbm.FBM_ERR_INVALID_ARG),
                         (16, 0.0, fbm.FBM_ERR_INVALID_ARG), (5, 2, fbm.FBM_ERR_INVALID_ARG),
                         (18, None, fbm.FBM_ERR_INVALID_ARG)):
        a = list(f)
        a[i] = bad
        assert L.sparse_fmha_fwd_fp8(*a) == code, (i, bad)
    a = list(f)
    a[17], a[10] = 1, 512           # causal with s_q != s_k
    assert L.sparse_fmha_fwd_fp8(*a) == fbm.FBM_ERR_UNSUPPORTED


def test_partial_mode_needs_both_partial_buffers(L):
    assert _fm(L, out=None, op=FAKE, lp=None) == fbm.FBM_ERR_INVALID_ARG
    assert _fm(L, out=None, op=None, lp=FAKE) == fbm.FBM_ERR_INVALID_ARG


def test_kernel_kind_is_host_only(L):
    assert L.fbm_fmha_kernel_kind(0, 96, 96, 1, 128, 128) == 0
    assert L.fbm_fmha_kernel_kind(1, 64, 64, 2, 128, 128) == 1
    assert L.fbm_fmha_kernel_kind(1, 128, 128, 1, 16384, 16384) in (1, 2)


def test_static_block_map_rejects_oversized_shapes_on_the_host(L):
    # b2 hq64 s32768 d128 needs more scratch than the static array holds
    need = fbm.block_map_workspace_bytes(2, 64, 64, 32768, 128)
    assert need > fbm.FBM_STATIC_SCRATCH_BYTES
    arr = (ctypes.c_float * 64)(*([0.1] * 64))
    st = L.sparge_block_map_static(FAKE, FAKE, 0, 2, 64, 64, 32768, 128, 64, 64, arr, None, arr,
                                   0.08, 0, 0, 0, FAKE, FAKE, None, None)
    assert st == fbm.FBM_ERR_UNSUPPORTED
    assert b"static array" in L.fbm_last_error_message()


def test_static_block_map_holds_the_headline_shape(L):
    # b2 h32 s16384 d128 (with its K-smoothing row) fits in the static array,
    # as do the causal GQA shape b1 hq32 hk8 s32768 and a tiny one
    for shape in ((2, 32, 32, 16384, 128), (1, 32, 8, 32768, 128), (1, 2, 2, 512, 64)):
        need = L.fbm_block_map_workspace_bytes(*shape, 64, 64)
        assert 0 < need <= fbm.FBM_STATIC_SCRATCH_BYTES, (shape, need)


def test_selftest_checks_its_limit_on_the_host(L):
    assert L.fbm_selftest_wait_timeout(0, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.fbm_selftest_wait_timeout(20_000_000_000, None) == fbm.FBM_ERR_INVALID_ARG


def test_fused_e4m3_block_map_checks_on_the_host(L):
    arr = (ctypes.c_float * 4)(*([0.1] * 4))
    args = [FAKE, FAKE, 0, 1, 4, 4, 1024, 128, 64, 64, arr, None, arr, 0.08, 0, 0, 0, FAKE, FAKE,
            None, FAKE, 1 << 30]
    # d = 64 is not supported (the codes feed the d = 128 fp8 attention)
    a = list(args)
    a[7] = 64
    assert L.sparge_block_map_e4m3(*a, FAKE, FAKE, FAKE, FAKE, None) == fbm.FBM_ERR_UNSUPPORTED
    # every code and scale buffer is required, the code buffers 16-byte aligned
    assert L.sparge_block_map_e4m3(*args, None, FAKE, FAKE, FAKE, None) == fbm.FBM_ERR_INVALID_ARG
    assert L.sparge_block_map_e4m3(*args, FAKE, FAKE, FAKE, None, None) == fbm.FBM_ERR_INVALID_ARG
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert L.sparge_block_map_e4m3(*args, odd, FAKE, FAKE, FAKE, None) == fbm.FBM_ERR_INVALID_ARG
