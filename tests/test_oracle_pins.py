"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test ties one oracle function to something other than itself:
a hand-worked case, brute-force token scoring, an independent sort, the
textbook dense / masked attention of ``torch`` (fp64), a stable argsort,
closed forms and the invariants the pages state.
"""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from datagen import bf16_to_f64, f32_to_bf16_rne


def bf16(x):
    return f32_to_bf16_rne(np.asarray(x, np.float32))


def rand_bf16(shape, seed, tid):
    n = int(np.prod(shape))
    return datagen.host_normal(n, seed, tid).reshape(shape)


# --------------------------------------------------------------------------- hand-worked selection
def test_hand_worked_selection():
    """Eight tokens, Bk=2, k=2 (local + 1): scores are the first key coordinate / sqrt(2)."""
    N, Bk, k, d_I = 8, 2, 2, 2
    key0 = [3, 1, 0, 5, 2, 2, -1, 4]
    k_idx = bf16([[v, 0.0] for v in key0])
    q_idx = bf16(np.tile([[[1.0, 0.0]]], (N, 1, 1)))
    rows = np.arange(N)
    S = oracle.block_scores(q_idx, k_idx, rows, N, Bk)[:, 0, :] * math.sqrt(2)
    ninf = -np.inf
    # block maxima over j <= t: block b holds tokens 2b, 2b+1
    expect_S = np.array([
        [3, ninf, ninf, ninf],
        [3, ninf, ninf, ninf],
        [3, 0, ninf, ninf],
        [3, 5, ninf, ninf],
        [3, 5, 2, ninf],
        [3, 5, 2, ninf],
        [3, 5, 2, -1],   # local block 3 sees only token 6 (j <= t)
        [3, 5, 2, 4],
    ])
    np.testing.assert_allclose(S, expect_S, rtol=1e-15)
    blk, kth = oracle.select_blocks(q_idx, k_idx, rows, N, Bk, k)
    expect = [[0, -1], [0, -1], [1, 0], [1, 0], [2, 1], [2, 1], [3, 1], [3, 1]]
    assert blk[0].tolist() == expect
    # t = 7: non-local blocks 0,1,2 score 3,5,2 -> taken 5, first left out 3
    np.testing.assert_allclose(kth[0, 7] * math.sqrt(2), [5, 3], rtol=1e-15)


def test_hand_worked_tie_goes_to_lower_block():
    N, Bk, k = 8, 2, 2
    key0 = [5, 1, 0, 5, 2, 5, 0, 0]      # blocks 0, 1, 2 all reach 5
    k_idx = bf16([[v, 0.0] for v in key0])
    q_idx = bf16(np.tile([[[1.0, 0.0]]], (N, 1, 1)))
    blk, _ = oracle.select_blocks(q_idx, k_idx, np.arange(N), N, Bk, k)
    assert blk[0, 7].tolist() == [3, 0]
    blk3, _ = oracle.select_blocks(q_idx, k_idx, np.arange(N), N, Bk, 3)
    assert blk3[0, 7].tolist() == [3, 0, 1]


# --------------------------------------------------------------------------- pooling vs brute force
@pytest.mark.parametrize("N,Bk,G,d_I", [(300, 64, 2, 32), (257, 16, 3, 8), (128, 128, 1, 16)])
def test_pooling_matches_bruteforce(N, Bk, G, d_I):
    """Token scores materialised with a float64 matmul, masked j <= t, max per block."""
    q_idx = rand_bf16((N, G, d_I), 11, 1)
    k_idx = rand_bf16((N, d_I), 11, 2)
    rows = np.arange(N)
    S = oracle.block_scores(q_idx, k_idx, rows, N, Bk)
    Q = bf16_to_f64(q_idx)
    K = bf16_to_f64(k_idx)
    nb = (N + Bk - 1) // Bk
    s = np.einsum("tgc,jc->tgj", Q, K) / math.sqrt(d_I)
    causal = np.arange(N)[None, :] <= np.arange(N)[:, None]
    s = np.where(causal[:, None, :], s, -np.inf)
    pad = nb * Bk - N
    s = np.concatenate([s, np.full((N, G, pad), -np.inf)], axis=2)
    brute = s.reshape(N, G, nb, Bk).max(axis=3)
    np.testing.assert_allclose(S, brute, rtol=1e-12, atol=0)


# --------------------------------------------------------------------------- top-k vs sort
@pytest.mark.parametrize("N,Bk,k", [(1024, 64, 4), (700, 32, 7), (512, 16, 40)])
def test_topk_matches_independent_sort(N, Bk, k):
    G, d_I = 2, 16
    q_idx = rand_bf16((N, G, d_I), 21, 1)
    k_idx = rand_bf16((N, d_I), 21, 2)
    rows = np.arange(N)
    S = oracle.block_scores(q_idx, k_idx, rows, N, Bk)
    blk, kth = oracle.select_blocks(q_idx, k_idx, rows, N, Bk, k)
    for t in range(N):
        loc = t // Bk
        for g in range(G):
            cand = np.arange(loc)
            order = cand[np.lexsort((cand, -S[t, g, :loc]))]      # score desc, block asc
            want = [loc] + order[: k - 1].tolist()
            want += [-1] * (k - len(want))
            assert blk[g, t].tolist() == want, (t, g)
            if loc > k - 1:
                assert kth[g, t, 0] == S[t, g, order[k - 2]] and kth[g, t, 1] == S[t, g, order[k - 1]]


def test_selection_invariants_tiny_config():
    cfg = datagen.CONFIGS["tiny"]
    inp = datagen.prefill_host(cfg)
    rows = np.arange(cfg.N)
    blk, _ = oracle.select_blocks(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    for g in range(cfg.G):
        for t in range(cfg.N):
            loc = t // cfg.Bk
            row = blk[g, t].tolist()
            ids = [b for b in row if b >= 0]
            assert row[0] == loc                                   # local block forced, slot 0
            assert len(ids) == min(cfg.k, loc + 1)                 # set size
            assert all(b <= loc for b in ids)                      # nothing beyond the query's block
            assert len(set(ids)) == len(ids)                       # no duplicates
            assert row[len(ids):] == [-1] * (cfg.k - len(ids))     # padding at the tail


@pytest.mark.parametrize("name,N", [("tiny", None), ("needles_4k", 4096)])
def test_planted_needles_are_selected(name, N):
    if name == "tiny":
        cfg = datagen.CONFIGS["tiny"]
    else:
        cfg = datagen.make_config(name, N=N, H_q=8, H_kv=4, d=32, d_I=128, Bk=128, k=8, needles=6)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    nd = inp["needles"]
    rows = np.arange(cfg.N)
    blk, _ = oracle.select_blocks(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    masks = datagen.pick_masks(cfg, nd, rows, rows, datagen.TID["pick"])
    n_checked = 0
    for t in range(cfg.N):
        for g in range(cfg.G):
            sel = set(blk[g, t].tolist())
            for n in range(nd.m):
                if masks[t, g] >> n & 1:
                    assert int(nd.blocks[0, g, n]) in sel, (t, g, n)
                    n_checked += 1
    assert n_checked > cfg.N // 4


# --------------------------------------------------------------------------- attention vs torch
def _sdpa(q, K, V, mask, scale):
    """torch fp64 scaled_dot_product_attention per head with an explicit boolean mask [H, T, N]."""
    out = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=scale)
    scores = (q @ K.transpose(-1, -2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    return out, lse


def _gqa_tensors(q_u16, K_u16, V_u16, gs):
    q = torch.from_numpy(bf16_to_f64(q_u16)).permute(1, 0, 2)                    # [H, T, d]
    K = torch.from_numpy(bf16_to_f64(K_u16)).permute(1, 0, 2).repeat_interleave(gs, 0)
    V = torch.from_numpy(bf16_to_f64(V_u16)).permute(1, 0, 2).repeat_interleave(gs, 0)
    return q, K, V


@pytest.mark.parametrize("N,H_q,H_kv,d,Bk,k", [(1024, 4, 1, 64, 64, 4), (333, 6, 2, 32, 32, 3)])
def test_sparse_attention_matches_torch_masked_sdpa(N, H_q, H_kv, d, Bk, k):
    G, d_I, gs = H_kv, 16, H_q // H_kv
    q = rand_bf16((N, H_q, d), 31, 1)
    K = rand_bf16((N, H_kv, d), 31, 2)
    V = rand_bf16((N, H_kv, d), 31, 3)
    q_idx = rand_bf16((N, G, d_I), 31, 4)
    k_idx = rand_bf16((N, d_I), 31, 5)
    rows = np.arange(N)
    blk, _ = oracle.select_blocks(q_idx, k_idx, rows, N, Bk, k)
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle.sparse_attn(q, K, V, blk, rows, Bk, scale)
    # mask built independently from the sets: key j allowed iff its block is in the set and j <= t
    jb = np.arange(N) // Bk
    mask = np.zeros((H_q, N, N), bool)
    for g in range(G):
        allowed = np.zeros((N, (N + Bk - 1) // Bk), bool)
        for t in range(N):
            ids = blk[g, t][blk[g, t] >= 0]
            allowed[t, ids] = True
        mg = allowed[:, jb] & (np.arange(N)[None, :] <= np.arange(N)[:, None])
        mask[g * gs:(g + 1) * gs] = mg[None]
    qt, Kt, Vt = _gqa_tensors(q, K, V, gs)
    ref, ref_lse = _sdpa(qt, Kt, Vt, torch.from_numpy(mask), scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.permute(1, 0).numpy(), rtol=1e-12, atol=1e-12)


def test_dense_attention_matches_torch_causal():
    N, H_q, H_kv, d = 200, 4, 2, 16
    q = rand_bf16((N, H_q, d), 41, 1)
    K = rand_bf16((N, H_kv, d), 41, 2)
    V = rand_bf16((N, H_kv, d), 41, 3)
    scale = 0.3
    rows = np.arange(N)
    out, lse = oracle.dense_attn(q, K, V, rows, scale)
    qt, Kt, Vt = _gqa_tensors(q, K, V, H_q // H_kv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, is_causal=True, scale=scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    causal = torch.ones(N, N, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(((qt @ Kt.transpose(-1, -2)) * scale).masked_fill(~causal, -math.inf), -1)
    np.testing.assert_allclose(lse, ref_lse.permute(1, 0).numpy(), rtol=1e-12)


@pytest.mark.parametrize("N,Bk,k", [(512, 64, 8), (512, 64, 12), (300, 300, 1), (256, 256, 1)])
def test_budget_covering_all_blocks_is_dense(N, Bk, k):
    """k >= number of visible blocks (or Bk = N, k = 1): MSA equals dense causal GQA."""
    H_q, H_kv, d, d_I = 4, 2, 32, 16
    q = rand_bf16((N, H_q, d), 51, 1)
    K = rand_bf16((N, H_kv, d), 51, 2)
    V = rand_bf16((N, H_kv, d), 51, 3)
    q_idx = rand_bf16((N, H_kv, d_I), 51, 4)
    k_idx = rand_bf16((N, d_I), 51, 5)
    rows = np.arange(N)
    blk, _ = oracle.select_blocks(q_idx, k_idx, rows, N, Bk, k)
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle.sparse_attn(q, K, V, blk, rows, Bk, scale)
    ref, ref_lse = oracle.dense_attn(q, K, V, rows, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)


def test_uniform_scores_give_mean_and_log_count():
    """q = 0: every visible key weighs the same, out = mean of V over J and lse = ln |J|."""
    N, H_q, H_kv, d, Bk, k = 640, 2, 1, 8, 64, 3
    q = np.zeros((N, H_q, d), np.uint16)
    K = rand_bf16((N, H_kv, d), 61, 2)
    V = rand_bf16((N, H_kv, d), 61, 3)
    blk = np.full((1, N, k), -1, np.int32)
    rng = np.random.default_rng(5)
    for t in range(N):
        loc = t // Bk
        others = rng.permutation(loc)[: k - 1] if loc else []
        ids = [loc] + list(others)
        blk[0, t, : len(ids)] = ids
    rows = np.arange(N)
    out, lse = oracle.sparse_attn(q, K, V, blk, rows, Bk, 0.125)
    Vf = bf16_to_f64(V)[:, 0, :]
    for t in range(0, N, 7):
        ids = blk[0, t][blk[0, t] >= 0]
        J = [j for b in ids for j in range(b * Bk, min((b + 1) * Bk, t + 1))]
        assert abs(lse[t, 0] - math.log(len(J))) < 1e-13
        np.testing.assert_allclose(out[t, 1], Vf[J].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_empty_set_gives_zero_and_minus_inf():
    N, d = 64, 8
    q = rand_bf16((N, 1, d), 71, 1)
    K = rand_bf16((N, 1, d), 71, 2)
    V = rand_bf16((N, 1, d), 71, 3)
    blk = np.full((1, N, 2), -1, np.int32)
    out, lse = oracle.sparse_attn(q, K, V, blk, np.arange(N), 16, 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_first_block_rows_are_causal_attention_inside_block0():
    N, H_q, H_kv, d, Bk, k = 256, 2, 1, 16, 64, 4
    q = rand_bf16((N, H_q, d), 81, 1)
    K = rand_bf16((N, H_kv, d), 81, 2)
    V = rand_bf16((N, H_kv, d), 81, 3)
    q_idx = rand_bf16((N, H_kv, 8), 81, 4)
    k_idx = rand_bf16((N, 8), 81, 5)
    rows = np.arange(Bk)
    blk, _ = oracle.select_blocks(q_idx[:Bk], k_idx, rows, N, Bk, k)
    assert np.all(blk[:, :, 0] == 0) and np.all(blk[:, :, 1:] == -1)
    out, lse = oracle.sparse_attn(q[:Bk], K, V, blk, rows, Bk, 0.25)
    ref, ref_lse = oracle.dense_attn(q[:Bk], K[:Bk], V[:Bk], rows, 0.25)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- inversion
@pytest.mark.parametrize("N,Bk,k,G", [(1024, 64, 4, 1), (777, 32, 5, 3)])
def test_inversion_matches_stable_argsort_and_round_trips(N, Bk, k, G):
    d_I = 16
    q_idx = rand_bf16((N, G, d_I), 91, 4)
    k_idx = rand_bf16((N, d_I), 91, 5)
    rows = np.arange(N)
    blk, _ = oracle.select_blocks(q_idx, k_idx, rows, N, Bk, k)
    # also poke a few holes (-1) into slots >= 1
    blk = blk.copy()
    blk[:, ::5, k - 1] = -1
    row_ptr, entries, n_entries = oracle.invert_blocks(blk, Bk)
    nb = (N + Bk - 1) // Bk
    for g in range(G):
        flat = blk[g].reshape(-1)
        e = np.nonzero(flat >= 0)[0]
        order = np.argsort(flat[e], kind="stable")
        want_entries = e[order].astype(np.int32)
        want_rp = np.concatenate([[0], np.cumsum(np.bincount(flat[e], minlength=nb))]).astype(np.int32)
        assert n_entries[g] == len(e)
        np.testing.assert_array_equal(row_ptr[g], want_rp)
        np.testing.assert_array_equal(entries[g, : len(e)], want_entries)
        # round trip B* -> B
        back = np.full(N * k, -1, np.int32)
        for b in range(nb):
            for x in entries[g, row_ptr[g, b]: row_ptr[g, b + 1]]:
                assert back[x] == -1
                back[x] = b
        np.testing.assert_array_equal(back, flat)
        # ascending t within each block
        for b in range(nb):
            ts = entries[g, row_ptr[g, b]: row_ptr[g, b + 1]] // k
            assert np.all(np.diff(ts) > 0)


# --------------------------------------------------------------------------- decode
def test_decode_equals_prefill_row():
    cfg = datagen.make_config("dec_small", kind="decode", B=3, ctx=1000, H_q=4, H_kv=2, d=32, d_I=32, Bk=64, k=4,
                              needles=2)
    ctx_len = np.array([1000, 700, 65], np.int64)
    inp = datagen.decode_host(cfg, ctx_len)
    scale = 1.0 / math.sqrt(cfg.d)
    out, lse, blk, kth = oracle.decode(inp["q_t"], inp["q_idx_t"], inp["k_idx_cache"], inp["k_cache"],
                                       inp["v_cache"], ctx_len, cfg.Bk, cfg.k, scale)
    for b in range(cfg.B):
        n = int(ctx_len[b])
        row = np.array([n - 1])
        pb, _ = oracle.select_blocks(inp["q_idx_t"][b:b + 1], inp["k_idx_cache"][b, :n], row, n, cfg.Bk, cfg.k)
        np.testing.assert_array_equal(blk[b], pb[:, 0, :])
        po, pl = oracle.sparse_attn(inp["q_t"][b:b + 1], inp["k_cache"][b, :n], inp["v_cache"][b, :n], pb, row,
                                    cfg.Bk, scale)
        np.testing.assert_allclose(out[b], po[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[b], pl[0], rtol=1e-13)
    # the needles each query picked are selected
    nd = inp["needles"]
    for b in range(cfg.B):
        mk = datagen.pick_masks(cfg, nd, [b], [ctx_len[b] - 1], datagen.TID["pick_t"], s=b)[0]
        for g in range(cfg.G):
            for n in range(nd.m):
                if mk[g] >> n & 1:
                    assert int(nd.blocks[b, g, n]) in set(blk[b, g].tolist())


def test_oracle_rejects_bad_arguments():
    q = np.zeros((2, 1, 4), np.uint16)
    k = np.zeros((4, 4), np.uint16)
    with pytest.raises(RuntimeError):
        oracle.select_blocks(q, k, np.array([0, 9]), 4, 2, 2)   # row beyond N
