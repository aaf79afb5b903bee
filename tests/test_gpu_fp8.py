"""FP8 (E4M3) index path on the GPU against the oracle: the quantizer bit for bit, the selection under
the set contract on the decoded values, prefill and decode (contiguous and paged) end to end."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from parity import (bf16_tensor_to_f64, check_set_invariants, compare_attn, compare_sets, decode_attn_check,
                    decode_sets_check, e4m3_codes, gamma_rows_e4m3)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    from block_sparse_long_index_gb300 import msa as m
    return m


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("n,x_off,y_off", [(1, 0, 0), (7, 0, 0), (8, 0, 0), (1000003, 0, 0), (4099, 1, 0),
                                           (4099, 0, 3), (65536, 8, 8)])
@pytest.mark.parametrize("scale", [1.0, 0.3, 40.0])
def test_quantize_bit_exact(msa, n, x_off, y_off, scale):
    rng = np.random.default_rng(n + x_off)
    vals = rng.standard_normal(n + x_off) * rng.choice([1e-4, 1e-2, 1.0, 30.0, 1e3], n + x_off)
    vals[: min(16, n)] = [0.0, -0.0, 448.0, -448.0, 464.0, 1e30, -1e30, 2.0 ** -10, 2.0 ** -9, -2.0 ** -9,
                          2.0 ** -6, 1.0625, 1.1875, 0.0009765625, 240.0, 256.0][: min(16, n)]
    x = _bf16_bits(vals)
    xd = dev_u16(x)[x_off:]
    y = torch.full((n + y_off,), 0xAA, dtype=torch.uint8, device="cuda")
    msa.msa_quantize_e4m3(xd, n, scale, y[y_off:])
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    ref = oracle.e4m3_quantize(x[x_off:], scale)
    assert np.array_equal(got[y_off:], ref)
    assert np.all(got[:y_off] == 0xAA)  # nothing written before y


SELECT_CASES = [
    # name, N, H_q, H_kv, d, d_I, Bk, k, needles
    ("f8_ragged_bk64", 1000, 8, 4, 64, 64, 64, 5, 2),
    ("f8_ragged_bk128_gs8", 2100, 16, 2, 128, 128, 128, 4, 3),
    ("f8_short", 50, 2, 1, 64, 64, 64, 4, 0),
    ("f8_k1_local_only", 777, 4, 2, 128, 128, 128, 1, 0),
    ("f8_k32_wide", 4096, 8, 8, 64, 128, 64, 32, 4),
    ("f8_gs1_g3", 1536, 3, 3, 128, 64, 128, 6, 2),
]


def _select_fp8(msa, q8, k8, N, G, d_I, Bk, k):
    blk = torch.full((G, N, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.msa_select_blocks_workspace(N, G, d_I, Bk, k), dtype=torch.uint8, device="cuda")
    msa.msa_select_blocks_fp8(dev_u8(q8), dev_u8(k8), N, G, d_I, Bk, k, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    return blk.cpu().numpy()


@pytest.mark.parametrize("case", SELECT_CASES, ids=[c[0] for c in SELECT_CASES])
def test_select_fp8_parity(msa, case, parity_log):
    name, N, H_q, H_kv, d, d_I, Bk, k, m = case
    cfg = datagen.make_config(name, N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k, needles=m)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    q8, k8 = e4m3_codes(inp["q_idx"]), e4m3_codes(inp["k_idx"])
    rows = np.arange(N)
    gpu = _select_fp8(msa, q8, k8, N, cfg.G, d_I, Bk, k)
    check_set_invariants(gpu, rows, Bk, k)
    ora, kth = oracle.select_blocks_e4m3(q8, k8, rows, N, Bk, k)
    S = oracle.block_scores_e4m3(q8, k8, rows, N, Bk)
    rep = compare_sets(gpu, ora, kth, S=S, gamma=gamma_rows_e4m3(q8, k8, rows, d_I), rows=rows, Bk=Bk)
    parity_log(name, sets=rep)
    nd = inp["needles"]
    if nd.m:
        masks = datagen.pick_masks(cfg, nd, rows, rows, datagen.TID["pick"])
        for t in range(N):
            for g in range(cfg.G):
                for n in range(nd.m):
                    if masks[t, g] >> n & 1:
                        assert int(nd.blocks[0, g, n]) in set(gpu[g, t].tolist())


def test_prefill_fp8_equals_select_fp8_then_attend(msa):
    cfg = datagen.make_config("f8_pipe", N=3000, H_q=16, H_kv=4, d=128, d_I=128, Bk=128, k=6, needles=3)
    inp = datagen.prefill_host(cfg)
    q8, k8 = dev_u8(e4m3_codes(inp["q_idx"])), dev_u8(e4m3_codes(inp["k_idx"]))
    q, kk, vv = dev_u16(inp["q"]), dev_u16(inp["k"]), dev_u16(inp["v"])
    shp = msa.shape(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    ws = torch.empty(msa.msa_prefill_workspace(shp), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(cfg.d)
    blk1 = torch.empty((cfg.G, cfg.N, cfg.k), dtype=torch.int32, device="cuda")
    out1 = torch.empty((cfg.N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
    lse1 = torch.empty((cfg.H_q, cfg.N), dtype=torch.float32, device="cuda")
    msa.msa_prefill_fp8(q, kk, vv, q8, k8, shp, scale, blk1, out1, lse1, ws)
    assert msa.msa_check_device_error(ws) == 0
    blk2 = torch.empty_like(blk1)
    msa.msa_select_blocks_fp8(q8, k8, cfg.N, cfg.G, cfg.d_I, cfg.Bk, cfg.k, blk2, ws)
    out2, lse2 = torch.empty_like(out1), torch.empty_like(lse1)
    msa.msa_sparse_attn_fwd(q, kk, vv, blk2, shp, scale, out2, lse2, ws)
    assert msa.msa_check_device_error(ws) == 0
    assert torch.equal(blk1, blk2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    # the outputs against the oracle's attention on the GPU's sets
    rows = np.arange(cfg.N)
    ref, ref_lse = oracle.sparse_attn(inp["q"], inp["k"], inp["v"], blk1.cpu().numpy(), rows, cfg.Bk, scale)
    print(compare_attn(bf16_tensor_to_f64(out1), lse1.T.cpu().numpy().astype(np.float64), ref, ref_lse))


DECODE_CASES = [
    ("f8_dec_small", 3, 5000, 8, 4, 128, 64, 64, 5, 2, [5000, 4097, 70]),
    ("f8_dec_bk128", 2, 20000, 16, 8, 128, 128, 128, 16, 4, [20000, 13000]),
    ("f8_dec_tiny_ctx", 2, 300, 4, 1, 64, 64, 64, 4, 1, [1, 300]),
]


def _decode_oracle_sets(q8, k8, ctx_len, Bk, k):
    """The oracle's block sets of each sequence's query row t = ctx_len - 1: [B, G, k] and kth [B, G, 2]."""
    B, G, _ = q8.shape
    blk = np.empty((B, G, k), np.int32)
    kth = np.empty((B, G, 2))
    for b in range(B):
        t = int(ctx_len[b]) - 1
        o, kt = oracle.select_blocks_e4m3(q8[b:b + 1], k8[b, :t + 1], [t], t + 1, Bk, k)
        blk[b], kth[b] = o[:, 0], kt[:, 0]
    return blk, kth


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_fp8_parity(msa, case, parity_log):
    name, B, C, H_q, H_kv, d, d_I, Bk, k, m, ctx_len = case
    cfg = datagen.make_config(name, kind="decode", B=B, ctx=C, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k,
                              needles=m)
    ctx_len = np.asarray(ctx_len, np.int64)
    inp = datagen.decode_host(cfg, ctx_len)
    q8, k8 = e4m3_codes(inp["q_idx_t"]), e4m3_codes(inp["k_idx_cache"])
    shp = msa.shape(C, H_q, H_kv, d, d_I, Bk, k)
    ws = torch.empty(msa.msa_decode_workspace(B, shp), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H_q), dtype=torch.float32, device="cuda")
    blk = torch.empty((B, H_kv, k), dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    msa.msa_decode_fp8(dev_u16(inp["q_t"]), dev_u8(q8), dev_u8(k8), dev_u16(inp["k_cache"]), dev_u16(inp["v_cache"]),
                       torch.from_numpy(ctx_len.astype(np.int32)).cuda(), B, shp, scale, out, lse, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    gpu_blk = blk.cpu().numpy()
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, Bk, k)
    rep, ora_blk = decode_sets_check(gpu_blk, q8, k8, ctx_len, Bk, k, fp8=True)
    np.testing.assert_array_equal(ora_blk, _decode_oracle_sets(q8, k8, ctx_len, Bk, k)[0])
    rep_a = decode_attn_check(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), gpu_blk, inp["q_t"],
                              lambda b: (inp["k_cache"][b], inp["v_cache"][b]), ctx_len, Bk, scale)
    parity_log(name, sets=rep, attn=rep_a)
    nd = inp["needles"]
    for b in range(B):
        mk = datagen.pick_masks(cfg, nd, [b], [ctx_len[b] - 1], datagen.TID["pick_t"], s=b)[0]
        for g in range(H_kv):
            for n in range(nd.m):
                if mk[g] >> n & 1:
                    assert int(nd.blocks[b, g, n]) in set(gpu_blk[b, g].tolist())


@pytest.mark.parametrize("page", [16, 128])
def test_decode_paged_fp8_equals_contiguous(msa, page, parity_log):
    """msa_decode_paged_fp8 on randomly paged pools equals msa_decode_fp8 on the contiguous caches bit for bit,
    and its results meet the oracle on the logical caches (sets under the set contract, out/lse on the GPU's
    own sets)."""
    B, C, H_q, H_kv, d, d_I, Bk, k = 3, 4096, 16, 4, 128, 128, 128, 8
    cfg = datagen.make_config("f8_paged", kind="decode", B=B, ctx=C, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=Bk, k=k,
                              needles=2)
    ctx_len = np.array([4096, 2500, 130], np.int64)
    inp = datagen.decode_host(cfg, ctx_len)
    q8, k8 = e4m3_codes(inp["q_idx_t"]), e4m3_codes(inp["k_idx_cache"])
    mp = C // page
    rng = np.random.default_rng(page)
    n_pages = B * mp + 5
    perm = rng.permutation(n_pages)[:B * mp].reshape(B, mp).astype(np.int32)
    kip = np.zeros((n_pages, page, d_I), np.uint8)
    kp = np.zeros((n_pages, page, H_kv, d), np.uint16)
    vp = np.zeros((n_pages, page, H_kv, d), np.uint16)
    for b in range(B):
        for lp in range(mp):
            kip[perm[b, lp]] = k8[b, lp * page:(lp + 1) * page]
            kp[perm[b, lp]] = inp["k_cache"][b, lp * page:(lp + 1) * page]
            vp[perm[b, lp]] = inp["v_cache"][b, lp * page:(lp + 1) * page]
    shp = msa.shape(C, H_q, H_kv, d, d_I, Bk, k)
    lens = torch.from_numpy(ctx_len.astype(np.int32)).cuda()
    scale = 0.09
    res = []
    for paged in (False, True):
        ws = torch.empty(msa.msa_decode_workspace(B, shp), dtype=torch.uint8, device="cuda")
        out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H_q), dtype=torch.float32, device="cuda")
        blk = torch.empty((B, H_kv, k), dtype=torch.int32, device="cuda")
        if paged:
            msa.msa_decode_paged_fp8(dev_u16(inp["q_t"]), dev_u8(q8), dev_u8(kip), dev_u16(kp), dev_u16(vp),
                                     torch.from_numpy(perm).cuda(), mp, n_pages, page, lens, B, shp, scale, out, lse,
                                     blk, ws)
        else:
            msa.msa_decode_fp8(dev_u16(inp["q_t"]), dev_u8(q8), dev_u8(k8), dev_u16(inp["k_cache"]),
                               dev_u16(inp["v_cache"]), lens, B, shp, scale, out, lse, blk, ws)
        assert msa.msa_check_device_error(ws) == 0
        res.append((out.view(torch.int16).cpu(), lse.cpu(), blk.cpu()))
    for a, b in zip(*res):
        assert torch.equal(a, b)
    p_out, p_lse, p_blk = res[1]
    gpu_blk = p_blk.numpy()
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, Bk, k)
    rep, _ = decode_sets_check(gpu_blk, q8, k8, ctx_len, Bk, k, fp8=True)
    rep_a = decode_attn_check(p_out.view(torch.bfloat16).double().numpy(), p_lse.double().numpy(), gpu_blk,
                              inp["q_t"], lambda b: (inp["k_cache"][b], inp["v_cache"][b]), ctx_len, Bk, scale)
    parity_log("f8_paged_%d" % page, sets=rep, attn=rep_a)
