"""Comparison rules between the CUDA path and the fp64 oracle (test infrastructure).

Block sets (the selection contract):
  * exact set equality on every row whose oracle gap between the last block
    taken and the first left out is >= 1e-2 * |last taken| ("near-tie" rows are
    exempt from equality and counted);
  * strict validity on EVERY row: the GPU set must be a correct top-(k-1)
    within the fp32 error bound gamma of a block maximum, i.e. every block it
    took scores (in the oracle's fp64 S) at least max(score of any block it
    left out) - 2*gamma, with gamma = d_I * 2^-22 * |q| * max_j |k_j| / sqrt(d_I);
  * structural invariants (local at slot 0, set size, ids <= local, no
    duplicates, -1 padding at the tail).

Attention (outputs computed on the same block sets on both sides):
  |gpu - ref| <= 2e-2 + 1e-2 * |ref| elementwise for out and lse, cosine >= 0.9999.
"""
from __future__ import annotations

import math

import numpy as np

ATOL, RTOL, COS_MIN = 2e-2, 1e-2, 0.9999
NEAR_TIE_REL = 1e-2


def bf16_tensor_to_f64(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def check_set_invariants(blk, rows, Bk, k):
    """blk [G, R, k] int32 for query positions rows[R]."""
    G, R, _ = blk.shape
    for g in range(G):
        for i, t in enumerate(rows):
            loc = int(t) // Bk
            row = blk[g, i].tolist()
            ids = [b for b in row if b >= 0]
            assert row[0] == loc, ("local not at slot 0", g, t, row)
            assert len(ids) == min(k, loc + 1), ("set size", g, t, row)
            assert all(b <= loc for b in ids), ("block beyond local", g, t, row)
            assert len(set(ids)) == len(ids), ("duplicate", g, t, row)
            assert row[len(ids):] == [-1] * (k - len(ids)), ("padding", g, t, row)


def gamma_rows(q_idx_rows_f64, k_idx_f64, rows, d_I):
    """fp32 error bound of a block max per (row, group): [R, G]."""
    knorm = np.linalg.norm(k_idx_f64, axis=1)
    # max |k_j| over the visible prefix j <= t
    prefix_max = np.maximum.accumulate(knorm)
    qn = np.linalg.norm(q_idx_rows_f64, axis=2)  # [R, G]
    km = prefix_max[np.asarray(rows)]
    return d_I * 2.0 ** -22 * qn * km[:, None] / math.sqrt(d_I)


def compare_sets(gpu_blk, ora_blk, kth, S=None, gamma=None, rows=None, Bk=None):
    """Returns a report dict; raises AssertionError on a contract violation.

    gpu_blk, ora_blk: [G, R, k]; kth: [G, R, 2] oracle (last taken, first left out);
    S: optional oracle block scores [R, G, nb] for the strict validity check; gamma [R, G]."""
    G, R, k = ora_blk.shape
    last, nxt = kth[..., 0], kth[..., 1]
    with np.errstate(invalid="ignore"):
        gap = last - nxt
        near = gap < NEAR_TIE_REL * np.abs(last)
    near = np.where(np.isinf(nxt) | np.isinf(last), False, near)
    gs = np.sort(gpu_blk, axis=2)
    os_ = np.sort(ora_blk, axis=2)
    mismatch = np.any(gs != os_, axis=2)
    bad = mismatch & ~near
    report = dict(rows=int(G * R), mismatch=int(mismatch.sum()), near_tie=int(near.sum()),
                  mismatch_outside_near_tie=int(bad.sum()))
    strict_bad = 0
    if S is not None:
        for g in range(G):
            for i in range(R):
                if not mismatch[g, i]:
                    continue
                t = int(rows[i])
                loc = t // Bk
                chosen = [b for b in gpu_blk[g, i, 1:].tolist() if b >= 0]
                if not chosen:
                    strict_bad += 1
                    continue
                cand = np.arange(loc)
                left = np.setdiff1d(cand, chosen)
                if len(left) == 0:
                    continue
                lo = S[i, g, chosen].min()
                hi = S[i, g, left].max()
                if lo < hi - 2.0 * gamma[i, g]:
                    strict_bad += 1
        report["strict_invalid"] = strict_bad
    assert report["mismatch_outside_near_tie"] == 0, report
    if S is not None:
        assert strict_bad == 0, report
    return report


def compare_sets_lazy(gpu_blk, ora_blk, kth, q_idx_rows, k_idx, rows, N, Bk):
    """compare_sets with the oracle's block scores computed only for rows whose sets differ."""
    import oracle
    from datagen import bf16_to_f64
    G, R, k = ora_blk.shape
    mism_rows = np.nonzero(np.any(np.any(np.sort(gpu_blk, 2) != np.sort(ora_blk, 2), axis=2), axis=0))[0]
    if len(mism_rows) == 0:
        rep = compare_sets(gpu_blk, ora_blk, kth)
        rep["strict_invalid"] = 0  # no row differs, so none can be invalid
        return rep
    sub_rows = np.asarray(rows)[mism_rows]
    S = oracle.block_scores(q_idx_rows[mism_rows], k_idx, sub_rows, N, Bk)
    gam = gamma_rows(bf16_to_f64(q_idx_rows[mism_rows]), bf16_to_f64(k_idx), sub_rows, q_idx_rows.shape[2])
    rep = compare_sets(gpu_blk[:, mism_rows], ora_blk[:, mism_rows], kth[:, mism_rows], S=S, gamma=gam,
                       rows=sub_rows, Bk=Bk)
    full = compare_sets(gpu_blk, ora_blk, kth)
    full["strict_invalid"] = rep["strict_invalid"]
    return full


def compare_attn(out_gpu, lse_gpu, out_ref, lse_ref, mask=None):
    """out_*: [R, H, d]; lse_*: [R, H] (float64 arrays).  mask [R] selects rows to compare."""
    if mask is not None:
        out_gpu, lse_gpu, out_ref, lse_ref = out_gpu[mask], lse_gpu[mask], out_ref[mask], lse_ref[mask]
    err = np.abs(out_gpu - out_ref)
    tol = ATOL + RTOL * np.abs(out_ref)
    ok_out = bool(np.all(err <= tol))
    a, b = out_gpu.reshape(-1), out_ref.reshape(-1)
    na, nb_ = np.linalg.norm(a), np.linalg.norm(b)
    cos = float(a @ b / (na * nb_)) if na > 0 and nb_ > 0 else (1.0 if na == nb_ else 0.0)
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(inf_ref, np.isneginf(lse_gpu)), "-inf lse pattern differs"
    fin = ~inf_ref
    lerr = np.abs(lse_gpu[fin] - lse_ref[fin])
    ok_lse = bool(np.all(lerr <= ATOL + RTOL * np.abs(lse_ref[fin])))
    rep = dict(max_abs=float(err.max()) if err.size else 0.0,
               max_rel=float((err / np.maximum(np.abs(out_ref), 1e-30)).max()) if err.size else 0.0,
               cos=cos, lse_max_abs=float(lerr.max()) if lerr.size else 0.0, n=int(out_ref.shape[0]))
    assert ok_out, ("out outside 2e-2 abs + 1e-2 rel", rep)
    assert ok_lse, ("lse outside 2e-2 abs + 1e-2 rel", rep)
    assert cos >= COS_MIN, ("cosine below 0.9999", rep)
    return rep


def e4m3_codes(x_bf16_bits):
    """E4M3 codes (uint8) of bf16 values (uint16 bit patterns), cast by torch's float8_e4m3fn on the CPU:
    the FP8 index inputs of the tests, made independently of both the oracle and the CUDA path."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(x_bf16_bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def gamma_rows_e4m3(q_codes, k_codes, rows, d_I):
    """gamma_rows on the decoded values of E4M3 inputs."""
    import oracle
    return gamma_rows(oracle.e4m3_decode(q_codes), oracle.e4m3_decode(k_codes), rows, d_I)


def _sum_reports(reps):
    keys = ("rows", "mismatch", "near_tie", "mismatch_outside_near_tie", "strict_invalid")
    return {k_: int(sum(r.get(k_, 0) for r in reps)) for k_ in keys}


def decode_sets_check(gpu_blk, q_idx_t, k_idx_cache, ctx_len, Bk, k, fp8=False):
    """The selection contract on a decode step, sequence by sequence: set equality outside near-tie rows and,
    on every row whose set differs from the oracle's, the strict validity check against the oracle's fp64
    block scores (the same rules as prefill rows).

    gpu_blk [B, G, k]; q_idx_t [B, G, d_I] and k_idx_cache [B, ctx, d_I] as bf16 bit patterns (E4M3 codes
    with fp8=True).  Returns (summed report, oracle sets [B, G, k])."""
    import oracle
    from datagen import bf16_to_f64
    B, G, _ = gpu_blk.shape
    d_I = q_idx_t.shape[2]
    sel = oracle.select_blocks_e4m3 if fp8 else oracle.select_blocks
    scores = oracle.block_scores_e4m3 if fp8 else oracle.block_scores
    ora_all = np.empty_like(gpu_blk)
    reps = []
    for b in range(B):
        t = int(ctx_len[b]) - 1
        qb, kb = q_idx_t[b:b + 1], k_idx_cache[b, :t + 1]
        ora, kth = sel(qb, kb, [t], t + 1, Bk, k)
        ora_all[b] = ora[:, 0]
        g_b = gpu_blk[b][:, None, :]
        if np.array_equal(np.sort(g_b, 2), np.sort(ora, 2)):
            rep = compare_sets(g_b, ora, kth)
            rep["strict_invalid"] = 0
        else:
            S = scores(qb, kb, [t], t + 1, Bk)
            gam = gamma_rows_e4m3(qb, kb, [t], d_I) if fp8 else gamma_rows(bf16_to_f64(qb), bf16_to_f64(kb), [t], d_I)
            rep = compare_sets(g_b, ora, kth, S=S, gamma=gam, rows=[t], Bk=Bk)
        reps.append(rep)
    return _sum_reports(reps), ora_all


def decode_attn_check(out_gpu, lse_gpu, gpu_blk, q_t, kv_rows, ctx_len, Bk, scale):
    """out [B, H_q, d] and lse [B, H_q] (float64) of a decode step against the oracle's attention on the GPU's
    own block sets, for every (sequence, head).  kv_rows(b) gives sequence b's (k_cache, v_cache) rows
    [ctx, H_kv, d] as bf16 bit patterns; only the rows of the GPU's blocks are read."""
    import oracle
    B = gpu_blk.shape[0]
    refs, lrefs = [], []
    for b in range(B):
        t = int(ctx_len[b]) - 1
        kc, vc = kv_rows(b)
        ref, ref_lse = oracle.sparse_attn(q_t[b:b + 1], kc, vc, gpu_blk[b][:, None, :], [t], Bk, scale)
        refs.append(ref)
        lrefs.append(ref_lse)
    return compare_attn(out_gpu, lse_gpu, np.concatenate(refs), np.concatenate(lrefs))
