"""Pins of the oracle's backward (msa_ref_sparse_attn_bwd) against things other than itself (CPU only).

The oracle writes the analytic gradients out (dZ = P (dP - D); dL/dz_index =
w (p_index - p_teacher)).  Here the same losses are built as plain fp64
``torch`` forward code over dense masks and differentiated by autograd, and
checked against identities that hold for any inputs.  Losses (study note 4-2
and 4-3; Flash-MSA KL section): main = sum(O * dO); index = w * sum over
(t, g) of KL(teacher || index) with the teacher (mean of the group's main
probabilities) detached and the index branch seeing only q^I and k^I.
"""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from datagen import bf16_to_f64


def rand_bf16(shape, seed, tid):
    return datagen.host_normal(int(np.prod(shape)), seed, tid).reshape(shape)


def make_case(N, H_q, H_kv, d, d_I, Bk, k, seed):
    q = rand_bf16((N, H_q, d), seed, 1)
    kk = rand_bf16((N, H_kv, d), seed, 2)
    v = rand_bf16((N, H_kv, d), seed, 3)
    q_idx = rand_bf16((N, H_kv, d_I), seed, 4)
    k_idx = rand_bf16((N, d_I), seed, 5)
    dout = rand_bf16((N, H_q, d), seed, 6)
    blk, _ = oracle.select_blocks(q_idx, k_idx, np.arange(N), N, Bk, k)
    return q, kk, v, q_idx, k_idx, dout, blk


def masks(blk, N, Bk):
    """mask[g, t, j]: j in J(t, g) = tokens of the row's set with j <= t (a repeated id counts once)."""
    G, _, k = blk.shape
    m = np.zeros((G, N, N), bool)
    for g in range(G):
        for t in range(N):
            for b in set(int(x) for x in blk[g, t] if x >= 0):
                lo, hi = b * Bk, min((b + 1) * Bk, t + 1)
                if lo < hi:
                    m[g, t, lo:hi] = True
    return torch.from_numpy(m)


def autograd_grads(q, kk, v, q_idx, k_idx, dout, blk, Bk, scale, w):
    N, H_q, d = q.shape
    H_kv = kk.shape[1]
    gs = H_q // H_kv
    d_I = q_idx.shape[2]
    t64 = lambda a: torch.from_numpy(bf16_to_f64(a)).requires_grad_(True)  # noqa: E731
    Q, K, V, QI, KI = t64(q), t64(kk), t64(v), t64(q_idx), t64(k_idx)
    dO = torch.from_numpy(bf16_to_f64(dout))
    M = masks(blk, N, Bk)                                         # [G, N, N]
    Kh = K.repeat_interleave(gs, dim=1)                           # [N, H_q, d]
    Vh = V.repeat_interleave(gs, dim=1)
    z = scale * torch.einsum("thd,jhd->htj", Q, Kh)               # [H_q, N, N]
    Mh = M.repeat_interleave(gs, dim=0)
    z = z.masked_fill(~Mh, float("-inf"))
    P = torch.softmax(z, dim=-1)
    O = torch.einsum("htj,jhd->thd", P, Vh)
    loss = (O * dO).sum()
    teacher = P.detach().view(H_kv, gs, N, N).mean(dim=1)          # [G, N, N]
    zI = torch.einsum("tgc,jc->gtj", QI, KI) / math.sqrt(d_I)
    zI = zI.masked_fill(~M, float("-inf"))
    logpI = torch.log_softmax(zI, dim=-1)
    kl_terms = torch.where(teacher > 0, teacher * (torch.log(teacher.clamp_min(1e-300)) - logpI),
                           torch.zeros_like(teacher))
    kl = kl_terms.sum(dim=-1)                                     # [G, N]
    (loss + w * kl.sum()).backward()
    return {"dq": Q.grad.numpy(), "dk": K.grad.numpy(), "dv": V.grad.numpy(), "dq_idx": QI.grad.numpy(),
            "dk_idx": KI.grad.numpy(), "kl": kl.detach().numpy()}


@pytest.mark.parametrize("N,H_q,H_kv,d,d_I,Bk,k,w", [(96, 4, 2, 16, 8, 8, 3, 1.0), (130, 8, 2, 8, 16, 16, 2, 0.37),
                                                    (64, 2, 1, 8, 8, 8, 8, 2.0)])
def test_bwd_matches_autograd(N, H_q, H_kv, d, d_I, Bk, k, w):
    q, kk, v, q_idx, k_idx, dout, blk = make_case(N, H_q, H_kv, d, d_I, Bk, k, seed=N + k)
    scale = 1.0 / math.sqrt(d)
    got = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, scale, w, n_threads=4)
    ref = autograd_grads(q, kk, v, q_idx, k_idx, dout, blk, Bk, scale, w)
    for name in ("dq", "dk", "dv", "dq_idx", "dk_idx", "kl"):
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-11, err_msg=name)


def test_bwd_invariants():
    """Each row's probabilities sum to 1, so sum_j dk_j = 0 and sum_j dk^I_j = 0; sum_j dv_{j,g} is the sum of
    the group's dO rows; KL >= 0; the index gradients scale with the KL weight and vanish at weight 0."""
    N, H_q, H_kv, d, d_I, Bk, k = 256, 8, 2, 16, 16, 16, 4
    q, kk, v, q_idx, k_idx, dout, blk = make_case(N, H_q, H_kv, d, d_I, Bk, k, seed=7)
    scale = 1.0 / math.sqrt(d)
    a = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, scale, 1.0, n_threads=4)
    gs = H_q // H_kv
    assert np.abs(a["dk"].sum(axis=0)).max() < 1e-10
    assert np.abs(a["dk_idx"].sum(axis=0)).max() < 1e-10
    dO = bf16_to_f64(dout).reshape(N, H_kv, gs, d).sum(axis=(0, 2))
    np.testing.assert_allclose(a["dv"].sum(axis=0), dO, rtol=1e-10, atol=1e-10)
    assert a["kl"].min() >= -1e-12 and a["kl"].max() > 0
    b = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, scale, 2.5, n_threads=4)
    np.testing.assert_allclose(b["dq_idx"], 2.5 * a["dq_idx"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["dk_idx"], 2.5 * a["dk_idx"], rtol=1e-12, atol=1e-14)
    for name in ("dq", "dk", "dv", "kl"):  # the main branch and the KL value do not depend on the weight
        np.testing.assert_array_equal(b[name], a[name])
    z = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, scale, 0.0, n_threads=4)
    assert not z["dq_idx"].any() and not z["dk_idx"].any()


def test_bwd_row_chunking_does_not_change_the_result():
    """The oracle's per-thread accumulators (rows split into chunks) only reorder the sums."""
    N, H_q, H_kv, d, d_I, Bk, k = 200, 4, 2, 8, 8, 8, 5
    q, kk, v, q_idx, k_idx, dout, blk = make_case(N, H_q, H_kv, d, d_I, Bk, k, seed=3)
    a = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, 0.3, 1.0, n_threads=1)
    b = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, 0.3, 1.0, n_threads=16)
    for name in a:
        np.testing.assert_allclose(a[name], b[name], rtol=1e-12, atol=1e-13, err_msg=name)


def test_bwd_rows_mode_equals_full():
    """The row-local mode (dq, dq_idx, kl of listed positions) reproduces the full backward's rows exactly."""
    N, H_q, H_kv, d, d_I, Bk, k = 200, 4, 2, 8, 8, 8, 5
    q, kk, v, q_idx, k_idx, dout, blk = make_case(N, H_q, H_kv, d, d_I, Bk, k, seed=5)
    a = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, 0.3, 0.8, n_threads=4)
    rows = np.array([0, 7, 8, 150, 199, 42, 42])
    b = oracle.sparse_attn_bwd_rows(q, kk, v, q_idx, k_idx, blk, dout, rows, Bk, 0.3, 0.8, n_threads=3)
    np.testing.assert_array_equal(b["dq"], a["dq"][rows])
    np.testing.assert_array_equal(b["dq_idx"], a["dq_idx"][rows])
    np.testing.assert_array_equal(b["kl"], a["kl"][:, rows])
