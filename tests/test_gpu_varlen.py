"""Varlen prefill: several sequences in block-aligned runs of cells (msa_select_blocks_varlen,
msa_prefill_varlen).  Every sequence must get exactly what it gets alone: the oracle on that sequence
(block ids offset by its first block), and the single-sequence GPU calls bit for bit."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from parity import bf16_tensor_to_f64, check_set_invariants, compare_attn, compare_sets, gamma_rows
from datagen import bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    from block_sparse_long_index_gb300 import msa as m
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


CASES = [
    # name, lengths, extra cells, H_q, H_kv, d, d_I, Bk, k
    ("bk128_mixed", [700, 128, 1, 0, 2000, 333], 256, 8, 2, 128, 128, 128, 6),
    ("bk64_split_tiles", [64, 65, 1000, 5, 191], 0, 8, 4, 64, 64, 64, 5),
    ("one_sequence", [1500], 0, 4, 2, 128, 128, 128, 4),
    ("k1_local_only", [300, 500], 128, 4, 1, 64, 32, 64, 1),
]


def _layout(lengths, extra, Bk):
    from block_sparse_long_index_gb300.api import varlen_cells
    cu = varlen_cells(lengths, Bk)
    return cu, cu[-1] + extra


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_select_varlen(msa, case):
    name, lengths, extra, H_q, H_kv, d, d_I, Bk, k = case
    cu, N = _layout(lengths, extra, Bk)
    cfg = datagen.make_config("vl_" + name, N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k, needles=0)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    G = H_kv
    blk = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    qd, kd = dev(inp["q_idx"]), dev(inp["k_idx"])
    msa.msa_select_blocks_varlen(qd, kd, cu_d, len(lengths), N, G, d_I, Bk, k, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    gpu = blk.cpu().numpy()
    for s, n in enumerate(lengths):
        if n == 0:
            continue
        c0, b0 = cu[s], cu[s] // Bk
        rows = np.arange(n)
        got = gpu[:, c0:c0 + n].copy()
        rel = np.where(got >= 0, got - b0, got)
        check_set_invariants(rel, rows, Bk, k)
        qs, ks = inp["q_idx"][c0:c0 + n], inp["k_idx"][c0:c0 + n]
        ora, kth = oracle.select_blocks(qs, ks, rows, n, Bk, k)
        S = oracle.block_scores(qs, ks, rows, n, Bk)
        rep = compare_sets(rel, ora, kth, S=S, gamma=gamma_rows(bf16_to_f64(qs), bf16_to_f64(ks), rows, d_I), rows=rows,
                           Bk=Bk)
        print(name, "sequence", s, rep)
        # the same sequence alone through msa_select_blocks: identical sets
        alone = torch.full((G, n, k), -7, dtype=torch.int32, device="cuda")
        ws1 = torch.empty(msa.msa_select_blocks_workspace(n, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
        msa.msa_select_blocks(dev(qs), dev(ks), n, G, d_I, Bk, k, alone, ws1)
        assert msa.msa_check_device_error(ws1) == 0
        assert np.array_equal(alone.cpu().numpy(), rel)
    # cells past the last sequence keep their local block only
    for t in range(cu[-1], N):
        assert gpu[0, t, 0] == t // Bk and np.all(gpu[:, t, 1:] == -1)


@pytest.mark.parametrize("case", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_prefill_varlen_equals_each_sequence_alone(msa, case):
    name, lengths, extra, H_q, H_kv, d, d_I, Bk, k = case
    cu, N = _layout(lengths, extra, Bk)
    cfg = datagen.make_config("vlp_" + name, N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k, needles=0)
    inp = datagen.prefill_host(cfg)
    G = H_kv
    scale = 1.0 / math.sqrt(d)
    shp = msa.shape(N, H_q, H_kv, d, d_I, Bk, k)
    ws = torch.empty(msa.msa_prefill_varlen_workspace(shp), dtype=torch.uint8, device="cuda")
    blk = torch.empty((G, N, k), dtype=torch.int32, device="cuda")
    out = torch.empty((N, H_q, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((H_q, N), dtype=torch.float32, device="cuda")
    msa.msa_prefill_varlen(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["q_idx"]), dev(inp["k_idx"]),
                           torch.tensor(cu, dtype=torch.int32, device="cuda"), len(lengths), shp, scale, blk, out, lse,
                           ws)
    assert msa.msa_check_device_error(ws) == 0
    for s, n in enumerate(lengths):
        if n == 0:
            continue
        c0, b0 = cu[s], cu[s] // Bk
        sl = slice(c0, c0 + n)
        shp1 = msa.shape(n, H_q, H_kv, d, d_I, Bk, k)
        ws1 = torch.empty(msa.msa_prefill_workspace(shp1), dtype=torch.uint8, device="cuda")
        blk1 = torch.empty((G, n, k), dtype=torch.int32, device="cuda")
        out1 = torch.empty((n, H_q, d), dtype=torch.bfloat16, device="cuda")
        lse1 = torch.empty((H_q, n), dtype=torch.float32, device="cuda")
        msa.msa_prefill(dev(inp["q"][sl]), dev(inp["k"][sl]), dev(inp["v"][sl]), dev(inp["q_idx"][sl]),
                        dev(inp["k_idx"][sl]), shp1, scale, blk1, out1, lse1, ws1)
        assert msa.msa_check_device_error(ws1) == 0
        got = blk[:, sl]
        assert torch.equal(torch.where(got >= 0, got - b0, got), blk1)
        assert torch.equal(out[sl].view(torch.int16), out1.view(torch.int16))
        assert torch.equal(lse[:, sl], lse1)
        # and against the oracle's attention on the sequence alone
        ref, ref_lse = oracle.sparse_attn(inp["q"][sl], inp["k"][sl], inp["v"][sl], blk1.cpu().numpy(), np.arange(n),
                                          Bk, scale)
        compare_attn(bf16_tensor_to_f64(out1), lse1.T.cpu().numpy().astype(np.float64), ref, ref_lse)


@pytest.mark.parametrize("cu", [[0, 100, 256], [0, 128, 64], [0, 128, 8192], [128, 256]])
def test_select_varlen_bad_offsets_are_flagged(msa, cu):
    """Offsets that are not block multiples, decrease, pass N or do not start at 0: the error word is set and
    every cell keeps only its local block (no fault, no read outside cu_seqlens)."""
    N, G, d_I, Bk, k = 512, 2, 64, 128, 4
    cfg = datagen.make_config("vl_bad", N=N, H_q=4, H_kv=G, d=64, d_I=d_I, Bk=Bk, k=k, needles=0)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    blk = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
    msa.msa_select_blocks_varlen(dev(inp["q_idx"]), dev(inp["k_idx"]), torch.tensor(cu, dtype=torch.int32,
                                 device="cuda"), len(cu) - 1, N, G, d_I, Bk, k, blk, ws)
    assert msa.msa_check_device_error(ws) == msa.MSA_ERR_BAD_INDEX
    b = blk.cpu().numpy()
    t = np.arange(N)
    assert np.all(b[:, :, 0] == t // Bk) and np.all(b[:, :, 1:] == -1)
