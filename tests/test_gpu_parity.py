"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, at sizes the oracle
finishes in seconds: several tiles, ragged tails, edge cases."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from datagen import bf16_to_f64
from parity import (bf16_tensor_to_f64, check_set_invariants, compare_attn, compare_sets, decode_attn_check,
                    decode_sets_check, gamma_rows)

pytestmark = pytest.mark.gpu


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.fixture(scope="module")
def msa():
    from block_sparse_long_index_gb300 import msa as m
    return m


def run_select(msa, q_idx, k_idx, N, G, d_I, Bk, k):
    blk = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")  # poisoned
    ws = torch.empty(msa.msa_select_blocks_workspace(N, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
    msa.msa_select_blocks(dev_bf16(q_idx), dev_bf16(k_idx), N, G, d_I, Bk, k, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    return blk.cpu().numpy()


def run_attn(msa, q, kk, vv, blk, N, H_q, H_kv, d, d_I, Bk, k, scale):
    shp = msa.shape(N, H_q, H_kv, d, d_I, Bk, k)
    ws = torch.empty(msa.msa_sparse_attn_fwd_workspace(shp), dtype=torch.uint8, device="cuda")
    out = torch.full((N, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H_q, N), float("nan"), dtype=torch.float32, device="cuda")
    b = blk if isinstance(blk, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(blk, np.int32)).cuda()
    msa.msa_sparse_attn_fwd(dev_bf16(q) if not isinstance(q, torch.Tensor) else q,
                            dev_bf16(kk) if not isinstance(kk, torch.Tensor) else kk,
                            dev_bf16(vv) if not isinstance(vv, torch.Tensor) else vv, b, shp, scale, out, lse, ws)
    status = msa.msa_check_device_error(ws)
    return out, lse, status


PREFILL_CASES = [
    # name, N, H_q, H_kv, d, d_I, Bk, k, needles
    ("tiny", None, None, None, None, None, None, None, None),
    ("ragged_bk64", 1000, 8, 4, 64, 64, 64, 5, 2),
    ("ragged_bk128_gs8", 2100, 16, 2, 128, 128, 128, 4, 3),
    ("short_under_one_block", 50, 2, 1, 64, 32, 64, 4, 0),
    ("k1_local_only", 777, 4, 2, 128, 32, 128, 1, 0),
    ("k32_wide", 4096, 8, 8, 64, 128, 64, 32, 4),
    ("gs1_bk128", 1536, 4, 4, 128, 64, 128, 6, 2),
]


def make_cfg(case):
    name, N, H_q, H_kv, d, d_I, Bk, k, m = case
    if name == "tiny":
        return datagen.CONFIGS["tiny"]
    return datagen.make_config(name, N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k, needles=m)


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_select_parity_full_rows(msa, case, parity_log):
    cfg = make_cfg(case)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    rows = np.arange(cfg.N)
    gpu = run_select(msa, inp["q_idx"], inp["k_idx"], cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k)
    check_set_invariants(gpu, rows, cfg.Bk, cfg.k)
    ora, kth = oracle.select_blocks(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    S = oracle.block_scores(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk)
    gam = gamma_rows(bf16_to_f64(inp["q_idx"]), bf16_to_f64(inp["k_idx"]), rows, cfg.d_I)
    rep = compare_sets(gpu, ora, kth, S=S, gamma=gam, rows=rows, Bk=cfg.Bk)
    parity_log(cfg.name, sets=rep)
    # planted needles are always selected
    nd = inp["needles"]
    if nd.m:
        masks = datagen.pick_masks(cfg, nd, rows, rows, datagen.TID["pick"])
        for t in range(cfg.N):
            for g in range(cfg.G):
                for n in range(nd.m):
                    if masks[t, g] >> n & 1:
                        assert int(nd.blocks[0, g, n]) in set(gpu[g, t].tolist())


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_attention_parity_on_oracle_sets(msa, case, parity_log):
    cfg = make_cfg(case)
    inp = datagen.prefill_host(cfg)
    rows = np.arange(cfg.N)
    ora, _ = oracle.select_blocks(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    scale = 1.0 / math.sqrt(cfg.d)
    out, lse, status = run_attn(msa, inp["q"], inp["k"], inp["v"], ora, cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I,
                                cfg.Bk, cfg.k, scale)
    assert status == 0
    ref, ref_lse = oracle.sparse_attn(inp["q"], inp["k"], inp["v"], ora, rows, cfg.Bk, scale)
    rep = compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref, ref_lse)
    parity_log(cfg.name + " attention on oracle sets", attn=rep)


def test_pipeline_select_then_attend(msa, parity_log):
    """select -> attend on the GPU: the sets under the set contract (strict check on every differing row), and
    out/lse of every row and head against the oracle's attention on the GPU's own sets."""
    cfg = datagen.make_config("pipe", N=3000, H_q=16, H_kv=4, d=128, d_I=128, Bk=128, k=6, needles=3)
    inp = datagen.prefill_host(cfg)
    from block_sparse_long_index_gb300 import MsaPrefill
    run = MsaPrefill(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    out, lse, blk = run(dev_bf16(inp["q"]), dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev_bf16(inp["q_idx"]),
                        dev_bf16(inp["k_idx"]))
    assert run.device_status() == 0
    gpu_blk = blk.cpu().numpy()
    rows = np.arange(cfg.N)
    check_set_invariants(gpu_blk, rows, cfg.Bk, cfg.k)
    ora, kth = oracle.select_blocks(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    S = oracle.block_scores(inp["q_idx"], inp["k_idx"], rows, cfg.N, cfg.Bk)
    gam = gamma_rows(bf16_to_f64(inp["q_idx"]), bf16_to_f64(inp["k_idx"]), rows, cfg.d_I)
    rep = compare_sets(gpu_blk, ora, kth, S=S, gamma=gam, rows=rows, Bk=cfg.Bk)
    ref, ref_lse = oracle.sparse_attn(inp["q"], inp["k"], inp["v"], gpu_blk, rows, cfg.Bk, 1 / math.sqrt(cfg.d))
    rep_a = compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref, ref_lse)
    parity_log("pipe", sets=rep, attn=rep_a)


@pytest.mark.parametrize("N,H_q,H_kv,d,d_I,Bk,k", [(16384, 16, 4, 128, 128, 128, 8), (20000, 8, 2, 64, 64, 64, 5)])
def test_prefill_call_equals_separate_calls(msa, N, H_q, H_kv, d, d_I, Bk, k):
    """msa_prefill (both stages in one call) gives the same block sets, out and lse as
    msa_select_blocks followed by msa_sparse_attn_fwd, also on a ragged N with a partial last block."""
    cfg = datagen.make_config("slabs", N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k, needles=2)
    dev = datagen.prefill_device(cfg)
    shp = msa.shape(N, H_q, H_kv, d, d_I, Bk, k)
    scale = 1.0 / math.sqrt(d)
    G = H_kv
    ws_sel = torch.empty(msa.msa_select_blocks_workspace(N, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
    blk_ref = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(dev["q_idx"], dev["k_idx"], N, G, d_I, Bk, k, blk_ref, ws_sel)
    out_ref, lse_ref, status = run_attn(msa, dev["q"], dev["k"], dev["v"], blk_ref, N, H_q, H_kv, d, d_I, Bk, k,
                                        scale)
    assert status == 0
    ws = torch.empty(msa.msa_prefill_workspace(shp), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace
        blk = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")
        out = torch.full((N, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((H_q, N), float("nan"), dtype=torch.float32, device="cuda")
        msa.msa_prefill(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"], shp, scale, blk, out, lse, ws)
        assert msa.msa_check_device_error(ws) == 0
        assert torch.equal(blk, blk_ref)
        assert torch.equal(out, out_ref)
        assert torch.equal(lse, lse_ref)


def test_host_pipeline_matches_device_calls():
    """PrefillHostPipeline (copies overlapped with compute across steps, two device input sets) returns,
    for each of three steps with different inputs, exactly the device-path outputs of that step."""
    from block_sparse_long_index_gb300 import MsaPrefill
    from block_sparse_long_index_gb300.api import PrefillHostPipeline
    names = ("q", "k", "v", "q_idx", "k_idx")
    cfgs = [datagen.make_config("hostpipe%d" % i, index=200 + i, N=2048, H_q=8, H_kv=2, d=64, d_I=64, Bk=64, k=6,
                                needles=2)
            for i in range(3)]
    run = MsaPrefill(2048, 8, 2, 64, 64, 64, 6)
    hosts, refs = [], []
    for cfg in cfgs:
        dev = datagen.prefill_device(cfg, want=names)
        out, lse, _ = run(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"])
        refs.append((out.cpu(), lse.cpu()))
        hosts.append({n: dev[n].cpu().pin_memory() for n in names})
    houts = [{"out": torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory(),
              "lse": torch.empty(run.lse.shape, dtype=run.lse.dtype).pin_memory()} for _ in range(3)]
    PrefillHostPipeline(run)(hosts, houts)
    torch.cuda.synchronize()
    assert run.device_status() == 0
    for (ro, rl), h in zip(refs, houts):
        assert torch.equal(h["out"], ro)
        assert torch.equal(h["lse"], rl)


def test_attention_dense_special_case(msa):
    """k >= number of blocks: MSA equals dense causal GQA attention."""
    N, H_q, H_kv, d, Bk = 1100, 8, 2, 64, 64
    k = (N + Bk - 1) // Bk
    q = datagen.host_normal(N * H_q * d, 5, 1).reshape(N, H_q, d)
    kk = datagen.host_normal(N * H_kv * d, 5, 2).reshape(N, H_kv, d)
    vv = datagen.host_normal(N * H_kv * d, 5, 3).reshape(N, H_kv, d)
    blk = np.full((H_kv, N, k), -1, np.int32)
    for t in range(N):
        loc = t // Bk
        blk[:, t, 0] = loc
        blk[:, t, 1:loc + 1] = np.arange(loc)
    k_lim = min(k, 32)
    blk = blk[:, :, :k_lim] if k > 32 else blk
    if k > 32:
        pytest.skip("k > 32 unsupported")
    scale = 1 / math.sqrt(d)
    out, lse, status = run_attn(msa, q, kk, vv, blk, N, H_q, H_kv, d, 32, Bk, k, scale)
    assert status == 0
    ref, ref_lse = oracle.dense_attn(q, kk, vv, np.arange(N), scale)
    compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref, ref_lse)


def test_attention_empty_sets_and_future_blocks(msa):
    """Rows whose set holds only -1 give out = 0, lse = -inf; ids past local(t) add nothing."""
    N, H_q, H_kv, d, Bk, k = 640, 4, 2, 64, 64, 3
    q = datagen.host_normal(N * H_q * d, 6, 1).reshape(N, H_q, d)
    kk = datagen.host_normal(N * H_kv * d, 6, 2).reshape(N, H_kv, d)
    vv = datagen.host_normal(N * H_kv * d, 6, 3).reshape(N, H_kv, d)
    blk = np.full((H_kv, N, k), -1, np.int32)
    rng = np.random.default_rng(0)
    nb = N // Bk
    for t in range(N):
        if t % 5 == 0:
            continue  # empty row
        loc = t // Bk
        blk[:, t, 0] = loc
        blk[:, t, 1] = (loc + 1 + rng.integers(0, nb - 1)) % nb  # any other block, possibly a future one
        if t % 11 == 0:
            blk[:, t, 2] = loc  # a repeated id counts once
    scale = 0.2
    out, lse, status = run_attn(msa, q, kk, vv, blk, N, H_q, H_kv, d, 32, Bk, k, scale)
    assert status == 0
    ref, ref_lse = oracle.sparse_attn(q, kk, vv, blk, np.arange(N), Bk, scale)
    compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref, ref_lse)


@pytest.mark.parametrize("N,G,Bk,k", [(1024, 1, 64, 4), (3001, 3, 128, 7), (5000, 8, 64, 16)])
def test_invert_parity_bit_exact(msa, N, G, Bk, k):
    """GPU B* equals the oracle's CSR bit for bit, on seeded random sets with holes."""
    rng = np.random.default_rng(N + G)
    blk = np.full((G, N, k), -1, np.int32)
    for g in range(G):
        for t in range(N):
            loc = t // Bk
            n = min(k, loc + 1)
            ids = [loc] + list(rng.permutation(loc)[: n - 1]) if loc else [loc]
            if t % 7 == 3 and n > 1:
                ids = ids[:-1]
            blk[g, t, : len(ids)] = ids
    nb = (N + Bk - 1) // Bk
    d_blk = torch.from_numpy(blk).cuda()
    row_ptr = torch.full((G, nb + 1), -9, dtype=torch.int32, device="cuda")
    entries = torch.full((G, N * k), -9, dtype=torch.int32, device="cuda")
    n_ent = torch.full((G,), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.msa_invert_blocks_workspace(N, G, Bk, k), dtype=torch.uint8, device="cuda")
    msa.msa_invert_blocks(d_blk, N, G, Bk, k, row_ptr, entries, n_ent, ws)
    assert msa.msa_check_device_error(ws) == 0
    rp, en, ne = oracle.invert_blocks(blk, Bk)
    np.testing.assert_array_equal(row_ptr.cpu().numpy(), rp)
    np.testing.assert_array_equal(n_ent.cpu().numpy(), ne)
    e = entries.cpu().numpy()
    for g in range(G):
        np.testing.assert_array_equal(e[g, : ne[g]], en[g, : ne[g]])


def test_bad_block_ids_raise_device_error_and_are_skipped(msa):
    N, H_q, H_kv, d, Bk, k = 512, 2, 1, 64, 64, 3
    q = datagen.host_normal(N * H_q * d, 8, 1).reshape(N, H_q, d)
    kk = datagen.host_normal(N * H_kv * d, 8, 2).reshape(N, H_kv, d)
    vv = datagen.host_normal(N * H_kv * d, 8, 3).reshape(N, H_kv, d)
    blk = np.full((1, N, k), -1, np.int32)
    blk[0, :, 0] = np.arange(N) // Bk
    blk[0, 100, 1] = 10 ** 6    # out of range
    blk[0, 200, 2] = -5         # negative, not -1
    out, lse, status = run_attn(msa, q, kk, vv, blk, N, H_q, H_kv, d, 32, Bk, k, 0.125)
    assert status == msa.MSA_ERR_BAD_INDEX
    clean = blk.copy()
    clean[0, 100, 1] = -1
    clean[0, 200, 2] = -1
    ref, ref_lse = oracle.sparse_attn(q, kk, vv, clean, np.arange(N), Bk, 0.125)
    compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref, ref_lse)


DECODE_CASES = [
    ("dec_small", 3, 5000, 8, 4, 128, 64, 64, 5, 2, [5000, 4097, 70]),
    ("dec_bk128", 2, 20000, 16, 8, 128, 128, 128, 16, 4, [20000, 13000]),
    ("dec_tiny_ctx", 2, 300, 4, 1, 64, 32, 64, 4, 1, [1, 300]),
    # k - 1 = 19 candidates: the scan CTAs keep 32-entry lists
    ("dec_k20", 2, 9000, 8, 2, 64, 64, 64, 20, 2, [9000, 6100]),
    # k = 1: the local block only (no candidate lists)
    ("dec_k1", 2, 3000, 8, 2, 64, 64, 64, 1, 0, [3000, 1500]),
    # about 133 candidate blocks per scan CTA in the first sequence (the register lists; up to 128 a CTA
    # sorts its blocks across the warp) and about 112 in the second (the sort)
    ("dec_cta_lists", 2, 1300000, 1, 1, 64, 32, 64, 4, 1, [1300000, 1100000]),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_parity(msa, case, parity_log):
    """Decode: every sequence's sets under the set contract (strict check on differing rows), and out/lse of
    every (sequence, head) against the oracle's attention on the GPU's own sets."""
    name, B, C, H_q, H_kv, d, d_I, Bk, k, m, ctx_len = case
    cfg = datagen.make_config(name, kind="decode", B=B, ctx=C, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k,
                              needles=m)
    ctx_len = np.asarray(ctx_len, np.int64)
    inp = datagen.decode_host(cfg, ctx_len)
    from block_sparse_long_index_gb300 import MsaDecode
    run = MsaDecode(B, C, H_q, H_kv, d, d_I, Bk, k)
    scale = 1 / math.sqrt(d)
    out, lse, blk = run(dev_bf16(inp["q_t"]), dev_bf16(inp["q_idx_t"]), dev_bf16(inp["k_idx_cache"]),
                        dev_bf16(inp["k_cache"]), dev_bf16(inp["v_cache"]),
                        torch.from_numpy(ctx_len.astype(np.int32)).cuda(), scale)
    assert run.device_status() == 0
    _, _, ora_blk, _ = oracle.decode(inp["q_t"], inp["q_idx_t"], inp["k_idx_cache"], inp["k_cache"],
                                     inp["v_cache"], ctx_len, Bk, k, scale)
    gpu_blk = blk.cpu().numpy()
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, Bk, k)
    rep, sel_ora = decode_sets_check(gpu_blk, inp["q_idx_t"], inp["k_idx_cache"], ctx_len, Bk, k)
    np.testing.assert_array_equal(sel_ora, ora_blk)  # the oracle's decode row is its prefill row
    rep_a = decode_attn_check(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), gpu_blk, inp["q_t"],
                              lambda b: (inp["k_cache"][b], inp["v_cache"][b]), ctx_len, Bk, scale)
    parity_log(name, sets=rep, attn=rep_a)


def _paged(cache, page, n_extra, rng):
    """Scatter a contiguous [B, C, ...] cache into a page pool with a random page table (plus unused pages)."""
    B, C = cache.shape[:2]
    mp = C // page
    n_pages = B * mp + n_extra
    perm = torch.from_numpy(rng.permutation(n_pages)[:B * mp].astype(np.int64)).view(B, mp)
    pool = torch.zeros((n_pages, page) + tuple(cache.shape[2:]), dtype=cache.dtype, device=cache.device)
    pool[perm.to(cache.device)] = cache.view((B, mp, page) + tuple(cache.shape[2:]))
    return pool, perm.to(torch.int32).cuda(), mp, n_pages


@pytest.mark.parametrize("page", [16, 64, 128, 512])
def test_decode_paged_equals_contiguous(msa, page, parity_log):
    """msa_decode_paged on pools scattered by a random page table gives exactly msa_decode's results on the
    contiguous caches (same sets, out and lse), with ragged lengths that end inside a page and a block; and the
    paged results meet the oracle on the logical caches: sets under the set contract, out/lse on the GPU's own
    sets."""
    B, C, H_q, H_kv, d, d_I, Bk, k = 3, 4096, 16, 4, 128, 128, 128, 8
    cfg = datagen.make_config("paged", kind="decode", B=B, ctx=C, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k,
                              needles=2)
    ctx_len = np.array([4096, 3001, 77], np.int64)
    inp = datagen.decode_host(cfg, ctx_len)
    q_t, q_idx_t = dev_bf16(inp["q_t"]), dev_bf16(inp["q_idx_t"])
    kic, kc, vc = dev_bf16(inp["k_idx_cache"]), dev_bf16(inp["k_cache"]), dev_bf16(inp["v_cache"])
    lens = torch.from_numpy(ctx_len.astype(np.int32)).cuda()
    shp = msa.shape(C, H_q, H_kv, d, d_I, Bk, k)
    scale = 1 / math.sqrt(d)
    ws = torch.empty(msa.msa_decode_workspace(B, shp), dtype=torch.uint8, device="cuda")
    outs = []
    for paged in (False, True):
        out = torch.full((B, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H_q), float("nan"), dtype=torch.float32, device="cuda")
        blk = torch.full((B, H_kv, k), -7, dtype=torch.int32, device="cuda")
        if paged:
            rng = np.random.default_rng(page)
            kip, table, mp, n_pages = _paged(kic, page, 5, rng)
            rng = np.random.default_rng(page)  # the same table for the K/V pools
            kp, _, _, _ = _paged(kc, page, 5, rng)
            rng = np.random.default_rng(page)
            vp, _, _, _ = _paged(vc, page, 5, rng)
            msa.msa_decode_paged(q_t, q_idx_t, kip, kp, vp, table, mp, n_pages, page, lens, B, shp, scale, out, lse,
                                 blk, ws)
        else:
            msa.msa_decode(q_t, q_idx_t, kic, kc, vc, lens, B, shp, scale, out, lse, blk, ws)
        assert msa.msa_check_device_error(ws) == 0
        outs.append((out, lse, blk))
    (o0, l0, b0), (o1, l1, b1) = outs
    assert torch.equal(b0, b1)
    assert torch.equal(o0, o1)
    assert torch.equal(l0, l1)
    gpu_blk = b1.cpu().numpy()
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, Bk, k)
    rep, _ = decode_sets_check(gpu_blk, inp["q_idx_t"], inp["k_idx_cache"], ctx_len, Bk, k)
    rep_a = decode_attn_check(bf16_tensor_to_f64(o1), l1.cpu().numpy().astype(np.float64), gpu_blk, inp["q_t"],
                              lambda b: (inp["k_cache"][b], inp["v_cache"][b]), ctx_len, Bk, scale)
    parity_log("paged_%d" % page, sets=rep, attn=rep_a)


def test_decode_paged_bad_page_id_is_flagged(msa):
    """A page id outside the pool sets MSA_ERR_BAD_INDEX (page 0 is read instead; nothing faults)."""
    B, C, H_q, H_kv, d, d_I, Bk, k, page = 1, 1024, 8, 2, 64, 64, 64, 4, 64
    cfg = datagen.make_config("paged_bad", kind="decode", B=B, ctx=C, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k,
                              needles=0)
    dev = datagen.decode_device(cfg)
    mp = C // page
    table = torch.arange(mp, dtype=torch.int32, device="cuda").view(1, mp).clone()
    table[0, 3] = mp + 100  # beyond the pool of mp pages
    shp = msa.shape(C, H_q, H_kv, d, d_I, Bk, k)
    ws = torch.empty(msa.msa_decode_workspace(B, shp), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((B,), C, dtype=torch.int32, device="cuda")
    kip = dev["k_idx_cache"].view(mp, page, d_I)
    kp = dev["k_cache"].view(mp, page, H_kv, d)
    vp = dev["v_cache"].view(mp, page, H_kv, d)
    msa.msa_decode_paged(dev["q_t"], dev["q_idx_t"], kip, kp, vp, table, mp, mp, page, lens, B, shp, 0.125, out, None,
                         None, ws)
    assert msa.msa_check_device_error(ws) == msa.MSA_ERR_BAD_INDEX


def test_datagen_device_matches_host():
    """The in-place device generator reproduces the host generator bit for bit."""
    cfg = datagen.make_config("dgchk", N=4096, H_q=8, H_kv=2, d=64, d_I=128, Bk=128, k=8, needles=3)
    host = datagen.prefill_host(cfg)
    devi = datagen.prefill_device(cfg)
    for name in ("q", "k", "v", "q_idx", "k_idx"):
        a = devi[name].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(a, host[name]), name
