"""Pins of the oracle's warmup mode (msa_ref_warmup_index) against things other than itself (CPU only).

Warmup ("MSA" study note 4-4): the main branch is dense causal attention and
the index branch is trained by the KL against the full-context teacher.  The
oracle writes the analytic gradients out; here they are checked against
* fp64 torch autograd of the same loss over the dense causal mask;
* the sparse backward oracle (itself pinned by autograd) given block sets that
  hold every visible block, where the two supports coincide;
* identities: sum_j dk^I_j = 0 (each row's index and teacher probabilities sum
  to one), KL >= 0, linearity in the KL weight, and row mode = full mode.
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


def make_case(N, H_q, H_kv, d, d_I, seed):
    return (rand_bf16((N, H_q, d), seed, 1), rand_bf16((N, H_kv, d), seed, 2), rand_bf16((N, H_kv, d_I), seed, 4),
            rand_bf16((N, d_I), seed, 5))


def autograd_warmup(q, kk, q_idx, k_idx, scale, w):
    N, H_q, d = q.shape
    H_kv = kk.shape[1]
    gs = H_q // H_kv
    d_I = q_idx.shape[2]
    Q, K = torch.from_numpy(bf16_to_f64(q)), torch.from_numpy(bf16_to_f64(kk))
    QI = torch.from_numpy(bf16_to_f64(q_idx)).requires_grad_(True)
    KI = torch.from_numpy(bf16_to_f64(k_idx)).requires_grad_(True)
    causal = torch.ones(N, N, dtype=torch.bool).tril()
    z = scale * torch.einsum("thd,jhd->htj", Q, K.repeat_interleave(gs, dim=1)).masked_fill(~causal, float("-inf"))
    teacher = torch.softmax(z, dim=-1).view(H_kv, gs, N, N).mean(dim=1)       # [G, N, N], no gradient
    zI = (torch.einsum("tgc,jc->gtj", QI, KI) / math.sqrt(d_I)).masked_fill(~causal, float("-inf"))
    logpI = torch.log_softmax(zI, dim=-1)
    terms = torch.where(teacher > 0, teacher * (torch.log(teacher.clamp_min(1e-300)) - logpI),
                        torch.zeros_like(teacher))
    kl = terms.sum(dim=-1)                                                     # [G, N]
    (w * kl.sum()).backward()
    return {"kl": kl.detach().numpy(), "dq_idx": QI.grad.numpy(), "dk_idx": KI.grad.numpy()}


def close(a, b, tol=1e-9):
    return float(np.abs(a - b).max()) <= tol * max(1.0, float(np.abs(b).max()))


@pytest.mark.parametrize("N,H_q,H_kv,d,d_I,w", [(80, 4, 2, 16, 8, 1.0), (130, 8, 2, 8, 16, 0.37),
                                               (64, 2, 1, 8, 8, 2.0)])
def test_warmup_matches_autograd(N, H_q, H_kv, d, d_I, w):
    q, kk, q_idx, k_idx = make_case(N, H_q, H_kv, d, d_I, seed=N + d)
    scale = 1.0 / math.sqrt(d)
    got = oracle.warmup_index(q, kk, q_idx, k_idx, scale, w)
    ref = autograd_warmup(q, kk, q_idx, k_idx, scale, w)
    for name in ("kl", "dq_idx", "dk_idx"):
        assert close(got[name], ref[name]), name


@pytest.mark.parametrize("N,H_q,H_kv,d,d_I,Bk", [(300, 4, 2, 16, 16, 64), (257, 8, 4, 8, 8, 32)])
def test_warmup_equals_sparse_backward_with_every_block(N, H_q, H_kv, d, d_I, Bk):
    q, kk, q_idx, k_idx = make_case(N, H_q, H_kv, d, d_I, seed=7 * N)
    nb = (N + Bk - 1) // Bk
    blk = np.full((H_kv, N, nb), -1, np.int32)
    for t in range(N):
        loc = t // Bk
        blk[:, t, 0] = loc
        blk[:, t, 1:loc + 1] = np.arange(loc)
    v = rand_bf16((N, H_kv, d), 3, 3)
    dout = np.zeros((N, H_q, d), np.uint16)
    scale, w = 0.3, 0.8
    sp = oracle.sparse_attn_bwd(q, kk, v, q_idx, k_idx, blk, dout, Bk, scale, w)
    wu = oracle.warmup_index(q, kk, q_idx, k_idx, scale, w)
    for name in ("kl", "dq_idx", "dk_idx"):
        assert close(wu[name], sp[name], 1e-11), name


def test_warmup_identities_and_rows():
    N, H_q, H_kv, d, d_I = 200, 8, 2, 16, 16
    q, kk, q_idx, k_idx = make_case(N, H_q, H_kv, d, d_I, seed=11)
    full = oracle.warmup_index(q, kk, q_idx, k_idx, 0.25, 1.0)
    assert np.all(full["kl"] >= -1e-12)
    tot = full["dk_idx"].sum(axis=0)
    assert float(np.abs(tot).max()) <= 1e-10 * float(np.abs(full["dk_idx"]).max())
    half = oracle.warmup_index(q, kk, q_idx, k_idx, 0.25, 0.5)
    assert close(half["dq_idx"] * 2, full["dq_idx"], 1e-12) and close(half["kl"], full["kl"], 0)
    rows = np.array([0, 1, 63, 64, 150, 199])
    part = oracle.warmup_index(q, kk, q_idx, k_idx, 0.25, 1.0, rows=rows)
    assert part["dk_idx"] is None
    assert np.array_equal(part["kl"], full["kl"][:, rows])
    assert np.array_equal(part["dq_idx"], full["dq_idx"][rows])
    # row 0 sees only itself: both distributions are one-hot, KL = 0 and no gradient
    assert full["kl"][:, 0].max() == 0.0 and np.abs(full["dq_idx"][0]).max() == 0.0


def test_warmup_lse_idx_is_the_index_logsumexp():
    N, H_q, H_kv, d, d_I = 90, 4, 2, 8, 16
    q, kk, q_idx, k_idx = make_case(N, H_q, H_kv, d, d_I, seed=5)
    got = oracle.warmup_index(q, kk, q_idx, k_idx, 0.3, 1.0)["lse_idx"]
    zI = torch.einsum("tgc,jc->gtj", torch.from_numpy(bf16_to_f64(q_idx)), torch.from_numpy(bf16_to_f64(k_idx)))
    zI = (zI / math.sqrt(d_I)).masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    assert close(got, torch.logsumexp(zI, dim=-1).numpy(), 1e-12)
