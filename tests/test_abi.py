"""The C ABI library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA.
CPU only."""
import ctypes

import pytest

from paged_kv_cache_174_gb300 import build as pkg_build
from paged_kv_cache_174_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return ops.lib()


def test_exports_every_declared_symbol(lib):
    names = ops.declared_symbols()
    assert {"pa_reshape_and_cache", "pa_paged_attention", "pa_copy_blocks",
            "pa_workspace_size", "pa_check_device_errors", "pa_get_last_error",
            "pa_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert ops.version() >= 100


def _status(code):
    return ops.STATUS_NAMES[code]


def test_host_side_argument_checks(lib):
    L = lib
    vp = ctypes.c_void_p
    # negative sizes are rejected before any CUDA call
    assert _status(L.pa_reshape_and_cache(None, None, -1, None, None, 4, 16, 2, 64, None, None)) \
        == "PA_ERR_INVALID_ARG"
    assert b"num_tokens" in L.pa_get_last_error()
    # an empty call is a no-op
    assert L.pa_reshape_and_cache(None, None, 0, None, None, 4, 16, 2, 64, None, None) == 0
    assert _status(L.pa_copy_blocks(None, None, 0, 16, 2, 64, None, 0, None)) \
        == "PA_ERR_INVALID_ARG"
    assert L.pa_copy_blocks(None, None, 4, 16, 2, 64, None, 0, None) == 0
    assert _status(L.pa_copy_blocks(None, None, 4, 16, 2, 64, None, 3, None)) \
        == "PA_ERR_INVALID_ARG"
    # a token row must be a whole number of 16-byte vectors
    assert _status(L.pa_reshape_and_cache(None, None, 1, None, None, 4, 16, 1, 3, None, None)) \
        == "PA_ERR_UNSUPPORTED"
    args = dict(q=None, k=None, v=None, nb=32, bs=16, nq=4, nkv=2, d=64, bt=None, maxb=3,
                sl=None, qsl=None, S=4, T=4, mq=1, ms=48, scale=0.125, out=None, ws=None,
                wsb=0, st=None)

    def attn(**kw):
        a = {**args, **kw}
        return _status(L.pa_paged_attention(a["q"], a["k"], a["v"], a["nb"], a["bs"], a["nq"],
                                            a["nkv"], a["d"], a["bt"], a["maxb"], a["sl"],
                                            a["qsl"], a["S"], a["T"], a["mq"], a["ms"],
                                            ctypes.c_float(a["scale"]), a["out"], a["ws"],
                                            a["wsb"], a["st"]))
    assert attn(bs=64) == "PA_ERR_UNSUPPORTED"
    assert attn(bs=32) == "PA_ERR_INVALID_ARG"  # supported: stops at the null pointers
    assert attn(bs=32, nb=1 << 26) == "PA_ERR_UNSUPPORTED"  # 2^31 token slots
    assert attn(d=96) == "PA_ERR_UNSUPPORTED"
    assert attn(nq=6, nkv=4) == "PA_ERR_INVALID_ARG"
    assert attn(nq=48, nkv=2) == "PA_ERR_UNSUPPORTED"  # group 24
    assert attn(mq=5, ms=4) == "PA_ERR_INVALID_ARG"
    assert attn(scale=float("nan")) == "PA_ERR_INVALID_ARG"
    a = {**args, "mq": 2}
    assert _status(L.pa_paged_attention_qrange(
        a["q"], a["k"], a["v"], a["nb"], a["bs"], a["nq"], a["nkv"], a["d"], a["bt"], a["maxb"],
        a["sl"], a["qsl"], a["S"], a["T"], 3, a["mq"], a["ms"], ctypes.c_float(0.125), a["out"],
        a["ws"], a["wsb"], a["st"])) == "PA_ERR_INVALID_ARG"  # min_q_len > max_q_len
    assert b"min_q_len" in L.pa_get_last_error()
    assert attn(S=0) == "PA_OK"   # nothing to do
    assert attn() == "PA_ERR_INVALID_ARG"  # null pointers
    assert vp  # keep the import used
    # block swap
    assert L.pa_swap_staging_bytes(3, 16, 2, 64) == 2 * 3 * 16 * 2 * 64 * 2
    assert _status(L.pa_swap_out(None, None, 4, 16, 2, 64, None, -1, None, None, None, None)) \
        == "PA_ERR_INVALID_ARG"
    assert L.pa_swap_out(None, None, 4, 16, 2, 64, None, 0, None, None, None, None) == 0
    assert _status(L.pa_swap_in(None, None, 4, 16, 2, 64, None, 2, None, None, None, None)) \
        == "PA_ERR_INVALID_ARG"
    assert _status(L.pa_swap_in(None, None, 4, 16, 1, 3, None, 2, None, None, None, None)) \
        == "PA_ERR_UNSUPPORTED"


def test_torch_side_checks_without_gpu():
    import torch
    with pytest.raises((TypeError, ValueError)):
        ops.reshape_and_cache(torch.zeros(1, 2, 64), torch.zeros(1, 2, 64),
                              torch.zeros(4, 16, 2, 64), torch.zeros(4, 16, 2, 64),
                              torch.zeros(1, dtype=torch.int32))


def test_step_graph_argument_checks_without_gpu():
    """pa_step_graph_create rejects bad maxima before touching CUDA."""
    from paged_kv_cache_174_gb300.ops import StepBuffers
    L = ops.lib()
    b = StepBuffers()
    g = ctypes.c_void_p()
    assert _status(L.pa_step_graph_create(ctypes.byref(b), ctypes.byref(g))) \
        == "PA_ERR_INVALID_ARG"
    assert _status(L.pa_step_graph_create(None, ctypes.byref(g))) == "PA_ERR_INVALID_ARG"
    b.max_tokens, b.max_seqs, b.max_blocks, b.max_q_len, b.max_seq_len = 8, 2, 4, 8, 64
    b.max_pairs = 3  # copy_pairs left NULL
    assert _status(L.pa_step_graph_create(ctypes.byref(b), ctypes.byref(g))) \
        == "PA_ERR_INVALID_ARG"
    assert b"copy_pairs" in L.pa_get_last_error()
    assert L.pa_step_graph_destroy(None) == 0
    assert _status(L.pa_selftest_wait_timeout(0, None)) == "PA_ERR_INVALID_ARG"
    # the fused decode step needs its slot_mapping
    assert _status(L.pa_decode_step(None, None, None, None, None, 32, 16, 4, 2, 64, None, 3,
                                    None, None, 4, 4, 48, None, ctypes.c_float(0.125), None,
                                    None, 0, None)) == "PA_ERR_INVALID_ARG"
    assert _status(L.pa_selftest_wait_timeout(2_000_000_000, None)) == "PA_ERR_INVALID_ARG"


def test_fp8_page_format_host_checks(lib):
    """The 8-bit cache's page size, and the host-side checks of its calls
    (block_size a multiple of 16, head_dim 64 or 128), without a GPU."""
    L = lib
    assert L.pa_fp8_page_bytes(8, 128) == 16 * 8 * (128 + 4)
    assert L.pa_fp8_page_bytes(2, 64) == 16 * 2 * 68
    assert L.pa_fp8_page_bytes(0, 64) == 0 and L.pa_fp8_page_bytes(2, -1) == 0
    # a page is a whole number of 16-byte vectors for every shape
    for nkv in (1, 2, 3, 8):
        for d in (64, 128):
            assert L.pa_fp8_page_bytes(nkv, d) % 16 == 0
    assert _status(L.pa_reshape_and_cache_fp8(None, None, 1, None, None, 4, 8, 2, 64, None,
                                              None)) == "PA_ERR_UNSUPPORTED"  # block_size 8
    assert _status(L.pa_reshape_and_cache_fp8(None, None, 1, None, None, 4, 16, 2, 96, None,
                                              None)) == "PA_ERR_UNSUPPORTED"  # head_dim 96
    assert L.pa_reshape_and_cache_fp8(None, None, 0, None, None, 4, 16, 2, 64, None, None) == 0
    assert _status(L.pa_reshape_and_cache_fp8(None, None, 1, None, None, 4, 16, 2, 64, None,
                                              None)) == "PA_ERR_INVALID_ARG"  # null pointers
    assert _status(L.pa_copy_blocks_fp8(None, None, 4, 24, 2, 64, None, 1, None)) \
        == "PA_ERR_UNSUPPORTED"  # block_size 24
    assert L.pa_copy_blocks_fp8(None, None, 4, 48, 2, 64, None, 0, None) == 0
    assert _status(L.pa_copy_blocks_fp8(None, None, 4, 48, 2, 64, None, 1, None)) \
        == "PA_ERR_INVALID_ARG"


def test_fp8_cache_views_follow_the_page_format():
    """ops.fp8_cache_views reads a cache as the header lays it out: token row
    r of page p of block b is slot b * block_size + 16 p + r; its codes sit at
    (r * n_kv + h) * d in the page and its scales after all 16 rows' codes."""
    import numpy as np
    import torch
    nb, bs, nkv, d = 3, 32, 2, 64
    pb = ops.fp8_page_bytes(nkv, d)
    assert pb == 16 * nkv * (d + 4)
    raw = np.zeros((nb, bs // 16, pb), np.uint8)
    cb = 16 * nkv * d
    rng = np.random.default_rng(3)
    want_codes = rng.integers(0, 256, (nb * bs, nkv, d), dtype=np.uint8)
    want_scales = rng.standard_normal((nb * bs, nkv)).astype(np.float32)
    for slot in range(nb * bs):
        b, p, r = slot // bs, (slot % bs) // 16, slot % 16
        for h in range(nkv):
            raw[b, p, (r * nkv + h) * d:(r * nkv + h + 1) * d] = want_codes[slot, h]
            raw[b, p, cb + (r * nkv + h) * 4:cb + (r * nkv + h + 1) * 4] = \
                want_scales[slot, h:h + 1].view(np.uint8)
    codes, scales = ops.fp8_cache_views(torch.from_numpy(raw), nkv, d)
    assert tuple(codes.shape) == (nb, bs // 16, 16, nkv, d)
    assert tuple(scales.shape) == (nb, bs // 16, 16, nkv)
    assert np.array_equal(codes.numpy().reshape(-1, nkv, d), want_codes)
    assert np.array_equal(scales.numpy().reshape(-1, nkv), want_scales)
    with pytest.raises(ValueError):
        ops.fp8_cache_views(torch.from_numpy(raw), nkv + 1, d)  # another page size
