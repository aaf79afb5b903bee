"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle checks every row of the 32K prefill config, 512 seeded query rows
per head on the 128K and 1M prefill configs (always including t = 0, Bk-1, Bk,
N-1) and every sequence of the 1M decode config.  Outputs are compared on the
GPU's own block sets, on every checked row and head."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from parity import (bf16_tensor_to_f64, check_set_invariants, compare_attn, compare_sets, compare_sets_lazy,
                    decode_attn_check, decode_sets_check)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _prefill_sampled(name, parity_log, n_rows=512):
    """n_rows seeded rows per group (None: every row) of the prefill pipeline at full size: the sets under the
    set contract (strict check on every differing row), planted needles selected, the attention kernel on the
    oracle's sets, and the pipeline's out/lse of every checked row and head against the oracle's attention on
    the GPU's own sets."""
    from block_sparse_long_index_gb300 import MsaPrefill
    cfg = datagen.CONFIGS[name]
    dev = datagen.prefill_device(cfg)
    run = MsaPrefill(cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    out, lse, blk = run(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"])
    assert run.device_status() == 0
    if n_rows is None:
        rows = np.arange(cfg.N, dtype=np.int64)
    else:
        rows = datagen.sample_rows(cfg.N, n_rows, cfg.seed, must=(0, cfg.Bk - 1, cfg.Bk, cfg.N - 1))
    rows_d = torch.from_numpy(rows).cuda()
    gpu_blk = blk[:, rows_d].cpu().numpy()
    out_pipe = bf16_tensor_to_f64(out[rows_d])
    lse_pipe = lse[:, rows_d].T.cpu().numpy().astype(np.float64)
    host = datagen.prefill_host(cfg, rows=None if n_rows is None else rows)
    check_set_invariants(gpu_blk, rows, cfg.Bk, cfg.k)
    ora, kth = oracle.select_blocks(host["q_idx"], host["k_idx"], rows, cfg.N, cfg.Bk, cfg.k)
    rep = compare_sets_lazy(gpu_blk, ora, kth, host["q_idx"], host["k_idx"], rows, cfg.N, cfg.Bk)
    # needles picked by the checked rows are selected
    nd = host["needles"]
    masks = datagen.pick_masks(cfg, nd, rows, rows, datagen.TID["pick"])
    for i in range(len(rows)):
        for g in range(cfg.G):
            for n in range(nd.m):
                if masks[i, g] >> n & 1:
                    assert int(nd.blocks[0, g, n]) in set(gpu_blk[g, i].tolist())
    scale = 1.0 / math.sqrt(cfg.d)
    # (1) the attention kernel on the oracle's sets, at (up to 1024 of) the checked rows
    sub = np.arange(len(rows)) if len(rows) <= 1024 else np.sort(
        np.random.default_rng(cfg.seed).choice(len(rows), 1024, replace=False))
    sub_d = torch.from_numpy(rows[sub]).cuda()
    ref, ref_lse = oracle.sparse_attn(host["q"][sub], host["k"], host["v"],
                                      ora[:, sub], rows[sub], cfg.Bk, scale)
    blk2 = blk.clone()
    blk2[:, sub_d] = torch.from_numpy(np.ascontiguousarray(ora[:, sub])).cuda()
    out2, lse2 = run.attend(dev["q"], dev["k"], dev["v"], blk2)
    assert run.device_status() == 0
    rep2 = compare_attn(bf16_tensor_to_f64(out2[sub_d]), lse2[:, sub_d].T.cpu().numpy().astype(np.float64), ref,
                        ref_lse)
    del ref, ref_lse, out2, lse2, blk2
    # (2) the whole pipeline, every checked row and head, on the GPU's own sets
    ref_g, ref_g_lse = oracle.sparse_attn(host["q"], host["k"], host["v"], gpu_blk, rows, cfg.Bk, scale)
    rep3 = compare_attn(out_pipe, lse_pipe, ref_g, ref_g_lse)
    parity_log(name, sets=rep, attn_oracle_sets=rep2, attn=rep3)


def test_prefill_32k_full(parity_log):
    _prefill_sampled("prefill_32k", parity_log, n_rows=None)


def test_prefill_128k_sampled(parity_log):
    _prefill_sampled("prefill_128k", parity_log)


def test_prefill_1m_sampled(parity_log):
    _prefill_sampled("prefill_1m", parity_log)


def test_decode_1m_full(parity_log):
    """Every sequence of the 1M-context decode step: sets under the set contract (strict check on differing
    rows), needles selected, and out/lse of every (sequence, head) on the GPU's own sets."""
    from block_sparse_long_index_gb300 import MsaDecode
    cfg = datagen.CONFIGS["decode_1m"]
    dev = datagen.decode_device(cfg)
    run = MsaDecode(cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    scale = 1.0 / math.sqrt(cfg.d)
    out, lse, blk = run(dev["q_t"], dev["q_idx_t"], dev["k_idx_cache"], dev["k_cache"], dev["v_cache"],
                        dev["ctx_len"], scale)
    assert run.device_status() == 0
    gpu_blk = blk.cpu().numpy()
    ctx_len = dev["ctx_len_host"]
    host = datagen.decode_host(cfg, ctx_len, want=("q_t", "q_idx_t", "k_idx_cache"))
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, cfg.Bk, cfg.k)
    rep, _ = decode_sets_check(gpu_blk, host["q_idx_t"], host["k_idx_cache"], ctx_len, cfg.Bk, cfg.k)
    nd = host["needles"]
    for b in range(cfg.B):
        mk = datagen.pick_masks(cfg, nd, [b], [ctx_len[b] - 1], datagen.TID["pick_t"], s=b)[0]
        for g in range(cfg.G):
            for n in range(nd.m):
                if mk[g] >> n & 1:
                    assert int(nd.blocks[b, g, n]) in set(gpu_blk[b, g].tolist())
    rep_a = decode_attn_check(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), gpu_blk, host["q_t"],
                              lambda b: _decode_kv_rows(cfg, b, gpu_blk[b]), ctx_len, cfg.Bk, scale)
    parity_log("decode_1m", sets=rep, attn=rep_a)


def _decode_kv_rows(cfg, b, blocks):
    """Sequence b's K/V cache rows [ctx, H_kv, d] with only the listed blocks generated (the rest is zero and
    never read by the oracle's attention over those blocks)."""
    kc = np.zeros((cfg.ctx, cfg.H_kv, cfg.d), np.uint16)
    vc = np.zeros((cfg.ctx, cfg.H_kv, cfg.d), np.uint16)
    toks = np.concatenate([np.arange(x * cfg.Bk, min((x + 1) * cfg.Bk, cfg.ctx))
                           for x in sorted(set(np.asarray(blocks).reshape(-1).tolist())) if x >= 0])
    ids = b * cfg.ctx + toks
    kc[toks] = datagen.host_normal_rows(ids, cfg.H_kv * cfg.d, cfg.seed, datagen.TID["k_cache"]).reshape(
        -1, cfg.H_kv, cfg.d)
    vc[toks] = datagen.host_normal_rows(ids, cfg.H_kv * cfg.d, cfg.seed, datagen.TID["v_cache"]).reshape(
        -1, cfg.H_kv, cfg.d)
    return kc, vc


def _bwd_sampled(name, n_rows):
    """The backward at full size: dq, dq_idx and kl of sampled rows against the oracle (on the GPU's own sets,
    rules of test_gpu_bwd.py), and over every row the identities sum_j dk_j = 0, sum_j dk_idx_j = 0 and
    sum_j dv_{j,g} = the sum of the group's dout rows (each row's probabilities sum to 1)."""
    from test_gpu_bwd import rel_report
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.CONFIGS[name] if isinstance(name, str) else name
    N, G, d, d_I = cfg.N, cfg.G, cfg.d, cfg.d_I
    dev = datagen.prefill_device(cfg)
    dout = datagen.device_normal_(torch.empty((N, cfg.H_q, d), dtype=torch.bfloat16, device="cuda"), cfg.seed,
                                  datagen.TID["dout"])
    shp = msa.shape(N, cfg.H_q, cfg.H_kv, d, d_I, cfg.Bk, cfg.k)
    scale, w = 1.0 / math.sqrt(d), 1.0
    blk = torch.empty((G, N, cfg.k), dtype=torch.int32, device="cuda")
    out = torch.empty((N, cfg.H_q, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((cfg.H_q, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(msa.msa_prefill_workspace(shp), msa.msa_sparse_attn_bwd_workspace(shp)), dtype=torch.uint8,
                     device="cuda")
    msa.msa_prefill(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"], shp, scale, blk, out, lse, ws)
    f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device="cuda")  # noqa: E731
    g = dict(dq=f32(N, cfg.H_q, d), dk=f32(N, cfg.H_kv, d), dv=f32(N, cfg.H_kv, d), dq_idx=f32(N, G, d_I),
             dk_idx=f32(N, d_I), kl=f32(G, N))
    msa.msa_sparse_attn_bwd(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"], blk, out, lse, dout, shp, scale,
                            w, g["dq"], g["dk"], g["dv"], g["dq_idx"], g["dk_idx"], g["kl"], ws)
    assert msa.msa_check_device_error(ws) == 0
    # identities over every row (fp64 sums of the fp32 gradients)
    for nm, axis_shape in (("dk", (G, d)), ("dk_idx", (d_I,))):
        x = g[nm].double()
        tot = x.sum(dim=0).abs()
        norm = x.pow(2).sum(dim=0).sqrt()
        assert float((tot / norm).max()) < 2e-2, nm
    dv_sum = g["dv"].double().sum(dim=0)                                        # [G, d]
    do_sum = dout.double().view(N, G, cfg.gs, d).sum(dim=(0, 2))
    assert float(((dv_sum - do_sum).norm() / do_sum.norm())) < 1e-2
    # sampled rows against the oracle
    rows = datagen.sample_rows(N, n_rows, cfg.seed + 17, must=(0, cfg.Bk - 1, cfg.Bk, N - 1))
    rows_d = torch.from_numpy(rows).cuda()
    host = datagen.prefill_host(cfg, rows=rows, want=("q", "q_idx", "k", "v", "k_idx"))
    full = lambda part, shape: _scatter_rows(part, rows, shape)  # noqa: E731
    q_full = full(host["q"], (N, cfg.H_q, d))
    qi_full = full(host["q_idx"], (N, G, d_I))
    do_full = full(datagen.host_normal_rows(rows, cfg.H_q * d, cfg.seed, datagen.TID["dout"]).reshape(-1, cfg.H_q, d),
                   (N, cfg.H_q, d))
    ref = oracle.sparse_attn_bwd_rows(q_full, host["k"], host["v"], qi_full, host["k_idx"], blk.cpu().numpy(), do_full,
                                      rows, cfg.Bk, scale, w)
    reps = {}
    for nm, gpu in (("dq", g["dq"][rows_d]), ("dq_idx", g["dq_idx"][rows_d]), ("kl", g["kl"][:, rows_d])):
        reps[nm] = rel_report(gpu.cpu().numpy().astype(np.float64), ref[nm])
    print(name, "backward", reps)
    for nm, r in reps.items():
        assert r["ok"], (nm, r)


def _scatter_rows(part, rows, shape):
    full = np.zeros(shape, dtype=np.uint16)
    full[rows] = part
    return full


def test_bwd_32k_sampled():
    _bwd_sampled("prefill_32k", 256)


def test_bwd_128k_sampled():
    _bwd_sampled("prefill_128k", 64)


def test_bwd_two_query_slabs_sampled():
    """N above the backward's query-slab cap (131072 positions): two slabs, sampled rows from both."""
    cfg = datagen.make_config("bwd_two_slabs", N=180000, H_q=8, H_kv=2, d=128, d_I=128, Bk=128, k=8, needles=4)
    _bwd_sampled(cfg, 96)


def _device_e4m3(msa, x):
    y = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    msa.msa_quantize_e4m3(x, x.numel(), 1.0, y)
    return y


def test_select_fp8_128k_sampled(parity_log):
    """msa_select_blocks_fp8 at 128K on inputs cast by msa_quantize_e4m3 on the device; the oracle gets the
    torch CPU cast of the host inputs, and the two casts must agree byte for byte where they are compared."""
    from parity import e4m3_codes, gamma_rows_e4m3
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.CONFIGS["prefill_128k"]
    N, G = cfg.N, cfg.G
    dev = datagen.prefill_device(cfg, want=("q_idx", "k_idx"))
    q8, k8 = _device_e4m3(msa, dev["q_idx"]), _device_e4m3(msa, dev["k_idx"])
    del dev
    blk = torch.empty((G, N, cfg.k), dtype=torch.int32, device="cuda")
    ws = torch.empty(msa.msa_select_blocks_workspace(N, G, cfg.d_I, cfg.Bk, cfg.k), dtype=torch.uint8, device="cuda")
    msa.msa_select_blocks_fp8(q8, k8, N, G, cfg.d_I, cfg.Bk, cfg.k, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    rows = datagen.sample_rows(N, 512, cfg.seed, must=(0, cfg.Bk - 1, cfg.Bk, N - 1))
    rows_d = torch.from_numpy(rows).cuda()
    gpu_blk = blk[:, rows_d].cpu().numpy()
    host = datagen.prefill_host(cfg, rows=rows, want=("q_idx", "k_idx"))
    hq8, hk8 = e4m3_codes(host["q_idx"]), e4m3_codes(host["k_idx"])
    assert np.array_equal(q8[rows_d].cpu().numpy(), hq8)
    assert np.array_equal(k8.cpu().numpy(), hk8)
    check_set_invariants(gpu_blk, rows, cfg.Bk, cfg.k)
    ora, kth = oracle.select_blocks_e4m3(hq8, hk8, rows, N, cfg.Bk, cfg.k)
    mism = np.nonzero(np.any(np.any(np.sort(gpu_blk, 2) != np.sort(ora, 2), axis=2), axis=0))[0]
    rep = compare_sets(gpu_blk, ora, kth)
    if len(mism):
        S = oracle.block_scores_e4m3(hq8[mism], hk8, rows[mism], N, cfg.Bk)
        sub = compare_sets(gpu_blk[:, mism], ora[:, mism], kth[:, mism], S=S,
                           gamma=gamma_rows_e4m3(hq8[mism], hk8, rows[mism], cfg.d_I), rows=rows[mism], Bk=cfg.Bk)
        rep["strict_invalid"] = sub["strict_invalid"]
    parity_log("prefill_128k fp8", sets=rep)
    nd = host["needles"]
    masks = datagen.pick_masks(cfg, nd, rows, rows, datagen.TID["pick"])
    for i in range(len(rows)):
        for g in range(G):
            for n in range(nd.m):
                if masks[i, g] >> n & 1:
                    assert int(nd.blocks[0, g, n]) in set(gpu_blk[g, i].tolist())


def test_decode_fp8_1m_full(parity_log):
    """msa_decode_fp8 on the 1M-context decode workload: every sequence's sets against the oracle on the torch
    CPU cast of the host caches (equal, byte for byte, to the device cast), and the outputs against the oracle's
    attention on the GPU's sets."""
    from parity import e4m3_codes
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.CONFIGS["decode_1m"]
    dev = datagen.decode_device(cfg)
    qi8, ki8 = _device_e4m3(msa, dev["q_idx_t"]), _device_e4m3(msa, dev["k_idx_cache"])
    del dev["k_idx_cache"]
    shp = msa.shape(cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    ws = torch.empty(msa.msa_decode_workspace(cfg.B, shp), dtype=torch.uint8, device="cuda")
    out = torch.empty((cfg.B, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((cfg.B, cfg.H_q), dtype=torch.float32, device="cuda")
    blk = torch.empty((cfg.B, cfg.H_kv, cfg.k), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(cfg.d)
    msa.msa_decode_fp8(dev["q_t"], qi8, ki8, dev["k_cache"], dev["v_cache"], dev["ctx_len"], cfg.B, shp, scale, out,
                       lse, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    gpu_blk = blk.cpu().numpy()
    ctx_len = dev["ctx_len_host"]
    host = datagen.decode_host(cfg, ctx_len, want=("q_t", "q_idx_t", "k_idx_cache"))
    hq8, hk8 = e4m3_codes(host["q_idx_t"]), e4m3_codes(host["k_idx_cache"])
    assert np.array_equal(qi8.cpu().numpy(), hq8)
    assert np.array_equal(ki8.cpu().numpy(), hk8)
    check_set_invariants(gpu_blk.transpose(1, 0, 2), ctx_len - 1, cfg.Bk, cfg.k)
    rep, _ = decode_sets_check(gpu_blk, hq8, hk8, ctx_len, cfg.Bk, cfg.k, fp8=True)
    rep_a = decode_attn_check(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), gpu_blk, host["q_t"],
                              lambda b: _decode_kv_rows(cfg, b, gpu_blk[b]), ctx_len, cfg.Bk, scale)
    parity_log("decode_1m fp8", sets=rep, attn=rep_a)
    nd = host["needles"]
    for b in range(cfg.B):
        mk = datagen.pick_masks(cfg, nd, [b], [ctx_len[b] - 1], datagen.TID["pick_t"], s=b)[0]
        for g in range(cfg.G):
            for n in range(nd.m):
                if mk[g] >> n & 1:
                    assert int(nd.blocks[b, g, n]) in set(gpu_blk[b, g].tolist())


def test_warmup_32k_sampled():
    """Warmup mode at N = 32K with the 128K prefill's head shapes: sampled rows of out, lse, lse^I, KL and dq^I
    against the oracle's row mode, and over every key the identity sum_j dk^I_j = 0."""
    from test_gpu_bwd import rel_report
    from block_sparse_long_index_gb300 import msa
    cfg = datagen.make_config("warmup_32k", N=32768, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=16, needles=0,
                              index=7)
    N, G = cfg.N, cfg.G
    dev = datagen.prefill_device(cfg)
    shp = msa.shape(N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device="cuda")  # noqa: E731
    out = torch.empty((N, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
    lse, lse_idx = f32(cfg.H_q, N), f32(G, N)
    dq_idx, dk_idx, kl = f32(N, G, cfg.d_I), f32(N, cfg.d_I), f32(G, N)
    scale, w = 1.0 / math.sqrt(cfg.d), 1.0
    msa.msa_warmup_fwd(dev["q"], dev["k"], dev["v"], dev["q_idx"], dev["k_idx"], shp, scale, out, lse, lse_idx)
    msa.msa_warmup_index_grad(dev["q"], dev["k"], dev["q_idx"], dev["k_idx"], lse, lse_idx, shp, scale, w, dq_idx,
                              dk_idx, kl)
    torch.cuda.synchronize()
    x = dk_idx.double()
    assert float((x.sum(dim=0).abs() / x.pow(2).sum(dim=0).sqrt()).max()) < 2e-2
    rows = datagen.sample_rows(N, 96, cfg.seed, must=(0, 1, 63, 64, N - 1))
    rows_d = torch.from_numpy(rows).cuda()
    host = datagen.prefill_host(cfg, rows=rows)
    ref_o, ref_l = oracle.dense_attn(host["q"], host["k"], host["v"], rows, scale)
    compare_attn(bf16_tensor_to_f64(out[rows_d]), lse[:, rows_d].T.cpu().numpy().astype(np.float64), ref_o, ref_l)
    q_full = _scatter_rows(host["q"], rows, (N, cfg.H_q, cfg.d))
    qi_full = _scatter_rows(host["q_idx"], rows, (N, G, cfg.d_I))
    ref = oracle.warmup_index(q_full, host["k"], qi_full, host["k_idx"], scale, w, rows=rows)
    lerr = np.abs(lse_idx[:, rows_d].cpu().numpy() - ref["lse_idx"])
    assert float(lerr.max()) <= 2e-2 + 1e-2 * float(np.abs(ref["lse_idx"]).max())
    reps = {nm: rel_report(g.cpu().numpy().astype(np.float64), ref[nm])
            for nm, g in (("kl", kl[:, rows_d]), ("dq_idx", dq_idx[rows_d]))}
    print("warmup_32k", reps)
    for nm, r in reps.items():
        assert r["ok"], (nm, r)
