"""The C-ABI library loads and exports every declared symbol; host-side validation (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    so = os.path.join(ROOT, "block_sparse_long_index_gb300", "libmsa.so")
    if not os.path.exists(so):
        import __graft_entry__
        __graft_entry__.build()
    from block_sparse_long_index_gb300 import msa
    return msa


def declared_functions():
    text = open(os.path.join(ROOT, "include", "msa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    raw = lib.raw()
    for n in names:
        assert hasattr(raw, n), n
    assert sorted(lib.EXPORTS) == names


def test_status_strings(lib):
    for s in range(7):
        assert lib.msa_status_string(s)
    assert "unknown" in lib.msa_status_string(99)


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first


def test_select_validation(lib):
    raw = lib.raw()
    big = 1 << 30
    assert raw.msa_select_blocks(None, FAKE, 1024, 1, 32, 64, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_select_blocks(FAKE, FAKE, 0, 1, 32, 64, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 1, 48, 64, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 1, 32, 96, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 1, 32, 64, 33, FAKE, FAKE, big, None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 65, 32, 64, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_UNSUPPORTED
    mis = ctypes.c_void_p((1 << 20) + 2)
    assert raw.msa_select_blocks(mis, FAKE, 1024, 1, 32, 64, 4, FAKE, FAKE, big, None) == lib.MSA_ERR_INVALID_ARGUMENT
    need = lib.msa_select_blocks_workspace(1024, 1, 32, 64, 4)
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 1, 32, 64, 4, FAKE, FAKE, need - 1,
                                 None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    assert raw.msa_select_blocks(FAKE, FAKE, 1024, 1, 32, 64, 4, FAKE, None, need, None) == lib.MSA_ERR_INVALID_ARGUMENT


def test_attention_and_decode_validation(lib):
    raw = lib.raw()
    s = lib.shape(4096, 8, 3, 128, 128, 128, 16)  # gs not an integer
    assert raw.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, 1 << 40,
                                   None) == lib.MSA_ERR_INVALID_ARGUMENT
    s = lib.shape(4096, 48, 3, 128, 128, 128, 16)  # gs = 16 unsupported
    assert raw.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, 1 << 40,
                                   None) == lib.MSA_ERR_UNSUPPORTED
    s = lib.shape(4096, 16, 2, 96, 128, 128, 16)  # d = 96 unsupported
    assert raw.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, 1 << 40,
                                   None) == lib.MSA_ERR_UNSUPPORTED
    s = lib.shape(4096, 16, 2, 128, 128, 128, 16)
    assert raw.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), -1.0, FAKE, FAKE, FAKE, 1 << 40,
                                   None) == lib.MSA_ERR_INVALID_ARGUMENT
    need = lib.msa_sparse_attn_fwd_workspace(s)
    assert need > 256
    assert raw.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, need - 256,
                                   None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    d = lib.shape(1 << 20, 64, 16, 128, 128, 128, 16)  # decode supports at most 8 groups
    assert raw.msa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(d), 0.1, FAKE, None, None, FAKE,
                          1 << 40, None) == lib.MSA_ERR_UNSUPPORTED
    d = lib.shape(1 << 20, 64, 8, 128, 128, 128, 16)
    assert raw.msa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.byref(d), 0.1, FAKE, None, None, FAKE,
                          1 << 40, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert lib.msa_decode_workspace(4, d) > 256


def test_invert_validation(lib):
    raw = lib.raw()
    assert raw.msa_invert_blocks(None, 100, 1, 64, 4, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == \
        lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_invert_blocks(FAKE, 100, 1, 64, 4, FAKE, FAKE, FAKE, FAKE, 1, None) == \
        lib.MSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.msa_invert_blocks_workspace(1 << 20, 8, 128, 16) > 256


def test_prefill_and_paged_decode_validation(lib):
    raw = lib.raw()
    s = lib.shape(4096, 16, 2, 128, 128, 128, 16)
    need = lib.msa_prefill_workspace(s)
    assert need >= lib.msa_sparse_attn_fwd_workspace(s)
    assert raw.msa_prefill(FAKE, FAKE, FAKE, None, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, FAKE, need,
                           None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, FAKE, need - 256,
                           None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    # paged decode: capacity = max_pages * page_size, page_size a multiple of 16
    d = lib.shape(64 * 128, 16, 2, 128, 128, 128, 8)
    ws = lib.msa_decode_workspace(2, d)
    args = lambda mp, npg, ps, wsb: (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, mp, npg, ps, FAKE, 2, ctypes.byref(d), 0.1,  # noqa
                                     FAKE, None, None, FAKE, wsb, None)
    assert raw.msa_decode_paged(*args(64, 200, 120, ws)) == lib.MSA_ERR_INVALID_ARGUMENT  # 120 % 16 != 0
    assert raw.msa_decode_paged(*args(32, 200, 128, ws)) == lib.MSA_ERR_INVALID_ARGUMENT  # 32 * 128 != N
    assert raw.msa_decode_paged(*args(64, 0, 128, ws)) == lib.MSA_ERR_INVALID_ARGUMENT    # empty pool
    assert raw.msa_decode_paged(*args(64, 200, 128, ws - 256)) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    big = lib.shape(64 * 128, 64, 16, 128, 128, 128, 8)  # more than 8 groups
    assert raw.msa_decode_paged(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 200, 128, FAKE, 2, ctypes.byref(big), 0.1,
                                FAKE, None, None, FAKE, 1 << 40, None) == lib.MSA_ERR_UNSUPPORTED


def test_fp8_entry_points_validation(lib):
    raw = lib.raw()
    # FP8 index inputs take d_I of 64 or 128 only
    ws = lib.msa_select_blocks_workspace(4096, 2, 32, 128, 16)
    assert raw.msa_select_blocks_fp8(FAKE, FAKE, 4096, 2, 32, 128, 16, FAKE, FAKE, ws, None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_select_blocks_fp8(None, FAKE, 4096, 2, 128, 128, 16, FAKE, FAKE, ws,
                                     None) == lib.MSA_ERR_INVALID_ARGUMENT
    s32 = lib.shape(4096, 16, 2, 128, 32, 128, 16)
    need = lib.msa_prefill_workspace(s32)
    assert raw.msa_prefill_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s32), 0.1, FAKE, FAKE, FAKE, FAKE, need,
                               None) == lib.MSA_ERR_UNSUPPORTED
    d32 = lib.shape(8192, 16, 2, 128, 32, 128, 8)
    assert raw.msa_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, ctypes.byref(d32), 0.1, FAKE, None, None, FAKE,
                              1 << 40, None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_decode_paged_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 200, 128, FAKE, 2, ctypes.byref(d32), 0.1,
                                    FAKE, None, None, FAKE, 1 << 40, None) == lib.MSA_ERR_UNSUPPORTED
    d = lib.shape(8192, 16, 2, 128, 128, 128, 8)
    wsd = lib.msa_decode_workspace(2, d)
    assert raw.msa_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, ctypes.byref(d), 0.1, FAKE, None, None, FAKE,
                              wsd - 256, None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    # quantize: negative size, null pointers with work to do, odd bf16 address, NaN scale
    assert raw.msa_quantize_e4m3(FAKE, -1, 1.0, FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_quantize_e4m3(None, 8, 1.0, FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_quantize_e4m3(ctypes.c_void_p((1 << 20) + 1), 8, 1.0, FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_quantize_e4m3(FAKE, 8, float("nan"), FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_quantize_e4m3(None, 0, 1.0, None, None) == lib.MSA_OK  # nothing to do


def test_varlen_validation(lib):
    raw = lib.raw()
    N, G, d_I, Bk, k = 4096, 2, 128, 128, 8
    ws = lib.msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k)
    assert ws >= lib.msa_select_blocks_workspace(N, G, d_I, Bk, k) + (N // Bk) * 4
    assert raw.msa_select_blocks_varlen(FAKE, FAKE, None, 2, N, G, d_I, Bk, k, FAKE, FAKE, ws,
                                        None) == lib.MSA_ERR_INVALID_ARGUMENT  # no cu_seqlens
    assert raw.msa_select_blocks_varlen(FAKE, FAKE, FAKE, 0, N, G, d_I, Bk, k, FAKE, FAKE, ws,
                                        None) == lib.MSA_ERR_INVALID_ARGUMENT  # S = 0
    assert raw.msa_select_blocks_varlen(FAKE, FAKE, ctypes.c_void_p((1 << 20) + 2), 2, N, G, d_I, Bk, k, FAKE, FAKE,
                                        ws, None) == lib.MSA_ERR_INVALID_ARGUMENT  # misaligned int32
    assert raw.msa_select_blocks_varlen(FAKE, FAKE, FAKE, 2, N, G, d_I, Bk, k, FAKE, FAKE, ws - 256,
                                        None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    s = lib.shape(N, 16, G, 128, d_I, Bk, k)
    need = lib.msa_prefill_varlen_workspace(s)
    assert need >= lib.msa_prefill_workspace(s)
    assert raw.msa_prefill_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, ctypes.byref(s), 0.1, FAKE, FAKE, FAKE, FAKE,
                                  need - 256, None) == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    assert raw.msa_prefill_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, ctypes.byref(s), -1.0, FAKE, FAKE, FAKE, FAKE,
                                  need, None) == lib.MSA_ERR_INVALID_ARGUMENT


def test_varlen_cells_helper():
    from block_sparse_long_index_gb300.api import varlen_cells
    assert varlen_cells([1, 128, 129, 0, 300], 128) == [0, 128, 256, 512, 512, 896]
    assert varlen_cells([64], 64) == [0, 64]


def test_warmup_validation(lib):
    raw = lib.raw()
    s = lib.shape(1000, 16, 2, 128, 128, 128, 16)
    args = lambda scale: (FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), scale, FAKE, FAKE, FAKE, None)  # noqa: E731
    assert raw.msa_warmup_fwd(*args(0.0)) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_warmup_fwd(None, *args(0.1)[1:]) == lib.MSA_ERR_INVALID_ARGUMENT
    bad = lib.shape(1000, 24, 2, 128, 128, 128, 16)  # gs = 12
    assert raw.msa_warmup_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(bad), 0.1, FAKE, FAKE, FAKE,
                              None) == lib.MSA_ERR_UNSUPPORTED
    assert raw.msa_warmup_index_grad(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, float("nan"), FAKE,
                                     FAKE, FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT
    assert raw.msa_warmup_index_grad(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, 1.0, FAKE,
                                     ctypes.c_void_p((1 << 20) + 8), FAKE, None) == lib.MSA_ERR_INVALID_ARGUMENT


def test_bwd_workspace_teacher_is_slab_bounded(lib):
    """The backward's teacher buffer (G k Bk 2 bytes a position) is sized for one query slab of at most
    131072 positions: past one slab the workspace grows linearly, by the per-entry and per-row buffers
    only (B* entries, index partials, D, lse^I: a few KB a position, against 32 KB for the teacher)."""
    def ws(N):
        return lib.msa_sparse_attn_bwd_workspace(lib.shape(N, 64, 8, 128, 128, 128, 16))
    a, b, c = ws(131072), ws(262144), ws(524288)
    per_pos = (b - a) / 131072
    assert 0 < per_pos < 8192, per_pos
    assert abs((c - b) - 2 * (b - a)) < (1 << 16)  # linear past the slab, up to alignment
    # below one slab the teacher grows with N as well
    small = (ws(65536) - ws(32768)) / 32768
    assert small > per_pos + 8 * 16 * 128 * 2 * 0.9


def test_decode_noalloc_size_edge(lib):
    """msa_decode_noalloc takes its scratch from a fixed 8 MiB array.  Its size check is msa_decode_workspace:
    the first batch past the edge is rejected before any launch (the batch at the edge runs on the GPU in
    tests/test_zz_no_alloc.py), and the sizes cross the edge between those two batches."""
    raw = lib.raw()
    limit = 8 << 20
    s = lib.shape(1024, 64, 8, 128, 128, 128, 32)
    sizes = {B: lib.msa_decode_workspace(B, s) for B in range(1, 33)}
    b_max = max(B for B, n in sizes.items() if n <= limit)
    assert all(sizes[B] <= limit for B in range(1, b_max + 1))
    assert sizes[b_max] <= limit < sizes[b_max + 1]
    status = raw.msa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, b_max + 1, ctypes.byref(s), 0.1, FAKE, None,
                                    None, None)
    assert status == lib.MSA_ERR_WORKSPACE_TOO_SMALL
    assert raw.msa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.byref(s), 0.1, FAKE, None, None,
                                  None) == lib.MSA_ERR_INVALID_ARGUMENT
