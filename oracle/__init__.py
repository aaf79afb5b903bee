"""ORACLE — test infrastructure only.

A plain, slow fp64 CPU statement of the MSA forward path and its backward (``msa_oracle.c``),
loaded through ctypes.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
never does, and the two share no code.  Inputs are bf16 bit patterns
(``uint16`` numpy arrays); outputs are float64 / int32 numpy arrays.

Every function states the passage it follows in ``msa_oracle.c``.  All parts
are pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``
(brute-force token scoring, an independent sort, the textbook dense attention
and masked attention of ``torch``, a stable argsort, hand-worked cases and
invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libmsa_oracle.so")
_lib = None


def build():
    """Compile the oracle with gcc (plain C, no GPU)."""
    src = os.path.join(_HERE, "msa_oracle.c")
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c99", "-o", _SO, src, "-lm"]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + p.stdout.decode())


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        lib = ctypes.CDLL(_SO)
        P, I64, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.msa_ref_block_scores.argtypes = [P, P, P, I64, I64, I, I, I, P, I]
        lib.msa_ref_select_blocks.argtypes = [P, P, P, I64, I64, I, I, I, I, P, P, I]
        lib.msa_ref_e4m3_decode.argtypes = [P, I64, P]
        lib.msa_ref_e4m3_quantize.argtypes = [P, I64, ctypes.c_float, P]
        lib.msa_ref_block_scores_e4m3.argtypes = [P, P, P, I64, I64, I, I, I, P, I]
        lib.msa_ref_select_blocks_e4m3.argtypes = [P, P, P, I64, I64, I, I, I, I, P, P, I]
        lib.msa_ref_warmup_index.argtypes = [P, P, P, P, P, I64, I64, I, I, I, I, D, D, P, P, P, P, I]
        lib.msa_ref_invert_blocks.argtypes = [P, I64, I, I, I, P, P, P]
        lib.msa_ref_sparse_attn.argtypes = [P, P, P, P, P, I64, I64, I, I, I, I, I, D, P, P, I]
        lib.msa_ref_dense_attn.argtypes = [P, P, P, P, I64, I64, I, I, I, D, P, P, I]
        lib.msa_ref_decode.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, I, I, I, D, P, P, P, P, I]
        lib.msa_ref_sparse_attn_bwd.argtypes = [P, P, P, P, P, P, P, I64, I, I, I, I, I, I, D, D, P, P, P, P, P, P,
                                                I]
        lib.msa_ref_sparse_attn_bwd_rows.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I, I, I, I, I, I, D, D, P, P,
                                                     P, I]
        for f in ("msa_ref_block_scores", "msa_ref_select_blocks", "msa_ref_invert_blocks",
                  "msa_ref_sparse_attn", "msa_ref_dense_attn", "msa_ref_decode", "msa_ref_sparse_attn_bwd",
                  "msa_ref_sparse_attn_bwd_rows"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def threads():
    return max(1, os.cpu_count() or 1)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError("%s failed with status %d" % (name, rc))


def block_scores(q_idx_rows, k_idx, rows, N, Bk, n_threads=None):
    """S[r, g, b] = max_{j in b, j <= t_r} q^I.k^I_j / sqrt(d_I) (-inf past local(t)).

    "MSA" study note, 2-3 "Fixed attention budget" (equations for s and S)."""
    q_idx_rows, k_idx, rows = _u16(q_idx_rows), _u16(k_idx), _i64(rows)
    n_rows, G, d_I = q_idx_rows.shape
    nb = (N + Bk - 1) // Bk
    S = np.empty((n_rows, G, nb), np.float64)
    _check(_load().msa_ref_block_scores(_p(q_idx_rows), _p(k_idx), _p(rows), n_rows, N, G, d_I, Bk, _p(S),
                                        n_threads or threads()), "msa_ref_block_scores")
    return S


def select_blocks(q_idx_rows, k_idx, rows, N, Bk, k, n_threads=None):
    """block_idx[g, r, :] (slot 0 local, then descending score, -1 padding) and
    kth[g, r, :] = (last taken, first left out) non-local block scores.

    "MSA" study note 2-3 / 3-4 / 3-5; chipsbuilder "Che cos'é MSA"; Flash-MSA
    "プロキシアテンション" (local block pinned to +inf)."""
    q_idx_rows, k_idx, rows = _u16(q_idx_rows), _u16(k_idx), _i64(rows)
    n_rows, G, d_I = q_idx_rows.shape
    blk = np.empty((G, n_rows, k), np.int32)
    kth = np.empty((G, n_rows, 2), np.float64)
    _check(_load().msa_ref_select_blocks(_p(q_idx_rows), _p(k_idx), _p(rows), n_rows, N, G, d_I, Bk, k, _p(blk),
                                         _p(kth), n_threads or threads()), "msa_ref_select_blocks")
    return blk, kth


def e4m3_decode(codes):
    """Values (fp64) of FP8 E4M3 codes (OCP 8-bit floating point specification, E4M3)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _check(_load().msa_ref_e4m3_decode(_p(codes), codes.size, _p(out)), "msa_ref_e4m3_decode")
    return out


def e4m3_quantize(x_bf16, scale=1.0):
    """E4M3 codes of the fp32 products (bf16 x) * scale: nearest, ties to even, saturated at 448."""
    x = _u16(x_bf16)
    codes = np.empty(x.shape, np.uint8)
    _check(_load().msa_ref_e4m3_quantize(_p(x), x.size, float(scale), _p(codes)), "msa_ref_e4m3_quantize")
    return codes


def block_scores_e4m3(q_idx_rows, k_idx, rows, N, Bk, n_threads=None):
    """block_scores on FP8 E4M3 index inputs (chipsbuilder "Co-Design Del Kernel": FP8 precision)."""
    q_idx_rows, k_idx = np.ascontiguousarray(q_idx_rows, np.uint8), np.ascontiguousarray(k_idx, np.uint8)
    rows = _i64(rows)
    n_rows, G, d_I = q_idx_rows.shape
    nb = (N + Bk - 1) // Bk
    S = np.empty((n_rows, G, nb), np.float64)
    _check(_load().msa_ref_block_scores_e4m3(_p(q_idx_rows), _p(k_idx), _p(rows), n_rows, N, G, d_I, Bk, _p(S),
                                             n_threads or threads()), "msa_ref_block_scores_e4m3")
    return S


def select_blocks_e4m3(q_idx_rows, k_idx, rows, N, Bk, k, n_threads=None):
    """select_blocks on FP8 E4M3 index inputs: the same rule on the exactly decoded scores."""
    q_idx_rows, k_idx = np.ascontiguousarray(q_idx_rows, np.uint8), np.ascontiguousarray(k_idx, np.uint8)
    rows = _i64(rows)
    n_rows, G, d_I = q_idx_rows.shape
    blk = np.empty((G, n_rows, k), np.int32)
    kth = np.empty((G, n_rows, 2), np.float64)
    _check(_load().msa_ref_select_blocks_e4m3(_p(q_idx_rows), _p(k_idx), _p(rows), n_rows, N, G, d_I, Bk, k,
                                              _p(blk), _p(kth), n_threads or threads()), "msa_ref_select_blocks_e4m3")
    return blk, kth


def invert_blocks(block_idx, Bk):
    """CSR B* per group: row_ptr [G, nb+1], entries [G, N*k] (t*k+slot, ascending t), n_entries [G].

    Flash-MSA "バックワードパス" (B -> B*)."""
    block_idx = np.ascontiguousarray(block_idx, np.int32)
    G, N, k = block_idx.shape
    nb = (N + Bk - 1) // Bk
    row_ptr = np.empty((G, nb + 1), np.int32)
    entries = np.full((G, N * k), -1, np.int32)
    n_entries = np.empty(G, np.int32)
    _check(_load().msa_ref_invert_blocks(_p(block_idx), N, G, Bk, k, _p(row_ptr), _p(entries), _p(n_entries)),
           "msa_ref_invert_blocks")
    return row_ptr, entries, n_entries


def sparse_attn(q_rows, K, V, block_idx_rows, rows, Bk, scale, n_threads=None):
    """out [n_rows, H_q, d] and lse [n_rows, H_q] over each row's selected blocks' tokens j <= t.

    "MSA" study note 2-3 (Attn over K_{g,B}, V_{g,B}) and 3-3 "Main Branch"."""
    q_rows, K, V, rows = _u16(q_rows), _u16(K), _u16(V), _i64(rows)
    block_idx_rows = np.ascontiguousarray(block_idx_rows, np.int32)
    n_rows, H_q, d = q_rows.shape
    N, H_kv, _ = K.shape
    k = block_idx_rows.shape[2]
    out = np.empty((n_rows, H_q, d), np.float64)
    lse = np.empty((n_rows, H_q), np.float64)
    _check(_load().msa_ref_sparse_attn(_p(q_rows), _p(K), _p(V), _p(block_idx_rows), _p(rows), n_rows, N, H_q,
                                       H_kv, d, Bk, k, float(scale), _p(out), _p(lse), n_threads or threads()),
           "msa_ref_sparse_attn")
    return out, lse


def dense_attn(q_rows, K, V, rows, scale, n_threads=None):
    """Dense causal GQA attention ("MSA" study note 1-1)."""
    q_rows, K, V, rows = _u16(q_rows), _u16(K), _u16(V), _i64(rows)
    n_rows, H_q, d = q_rows.shape
    N, H_kv, _ = K.shape
    out = np.empty((n_rows, H_q, d), np.float64)
    lse = np.empty((n_rows, H_q), np.float64)
    _check(_load().msa_ref_dense_attn(_p(q_rows), _p(K), _p(V), _p(rows), n_rows, N, H_q, H_kv, d, float(scale),
                                      _p(out), _p(lse), n_threads or threads()), "msa_ref_dense_attn")
    return out, lse


def decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, Bk, k, scale, n_threads=None):
    """One decode step: out [B,H_q,d], lse [B,H_q], block_idx [B,G,k], kth [B,G,2].

    velog llama.cpp analysis, section 2 (scan the whole index-key cache, read
    only the selected K/V blocks)."""
    q_t, q_idx_t, k_idx_cache = _u16(q_t), _u16(q_idx_t), _u16(k_idx_cache)
    k_cache, v_cache, ctx_len = _u16(k_cache), _u16(v_cache), _i64(ctx_len)
    B, H_q, d = q_t.shape
    _, G, d_I = q_idx_t.shape
    ctx_max = k_idx_cache.shape[1]
    H_kv = k_cache.shape[2]
    out = np.empty((B, H_q, d), np.float64)
    lse = np.empty((B, H_q), np.float64)
    blk = np.empty((B, G, k), np.int32)
    kth = np.empty((B, G, 2), np.float64)
    _check(_load().msa_ref_decode(_p(q_t), _p(q_idx_t), _p(k_idx_cache), _p(k_cache), _p(v_cache), _p(ctx_len), B,
                                  ctx_max, H_q, H_kv, d, d_I, Bk, k, float(scale), _p(out), _p(lse), _p(blk),
                                  _p(kth), n_threads or threads()), "msa_ref_decode")
    return out, lse, blk, kth


def sparse_attn_bwd(q, k, v, q_idx, k_idx, block_idx, dout, Bk, scale, kl_weight=1.0, n_threads=None):
    """Backward of the main branch (upstream dout) and of the index branch's KL loss over all N rows
    (msa_oracle.c: msa_ref_sparse_attn_bwd; study note 4-2 / 4-3, Flash-MSA KL section).  Inputs are
    bf16 bit patterns: q, dout [N, H_q, d]; k, v [N, H_kv, d]; q_idx [N, G, d_I]; k_idx [N, d_I];
    block_idx [G, N, k] int32.  Returns a dict of float64 arrays dq, dk, dv, dq_idx, dk_idx and kl [G, N]."""
    lib = _load()
    q, k, v, q_idx, k_idx, dout = (_u16(a) for a in (q, k, v, q_idx, k_idx, dout))
    blk = np.ascontiguousarray(block_idx, dtype=np.int32)
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    d_I = q_idx.shape[2]
    kk = blk.shape[2]
    out = {"dq": np.zeros((N, H_q, d)), "dk": np.zeros((N, H_kv, d)), "dv": np.zeros((N, H_kv, d)),
           "dq_idx": np.zeros((N, H_kv, d_I)), "dk_idx": np.zeros((N, d_I)), "kl": np.zeros((H_kv, N))}
    rc = lib.msa_ref_sparse_attn_bwd(_p(q), _p(k), _p(v), _p(q_idx), _p(k_idx), _p(blk), _p(dout), N, H_q, H_kv, d,
                                     d_I, Bk, kk, float(scale), float(kl_weight), _p(out["dq"]), _p(out["dk"]),
                                     _p(out["dv"]), _p(out["dq_idx"]), _p(out["dk_idx"]), _p(out["kl"]),
                                     n_threads or threads())
    _check(rc, "msa_ref_sparse_attn_bwd")
    return out


def sparse_attn_bwd_rows(q, k, v, q_idx, k_idx, block_idx, dout, rows, Bk, scale, kl_weight=1.0, n_threads=None):
    """The row-local backward outputs (dq [R, H_q, d], dq_idx [R, G, d_I], kl [G, R]) of the listed positions
    over full-size inputs (msa_oracle.c: msa_ref_sparse_attn_bwd_rows; same arithmetic as sparse_attn_bwd)."""
    lib = _load()
    q, k, v, q_idx, k_idx, dout = (_u16(a) for a in (q, k, v, q_idx, k_idx, dout))
    blk = np.ascontiguousarray(block_idx, dtype=np.int32)
    rows = _i64(rows)
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    d_I = q_idx.shape[2]
    R = len(rows)
    dq, dqi, kl = np.zeros((R, H_q, d)), np.zeros((R, H_kv, d_I)), np.zeros((H_kv, R))
    rc = lib.msa_ref_sparse_attn_bwd_rows(_p(q), _p(k), _p(v), _p(q_idx), _p(k_idx), _p(blk), _p(dout), _p(rows), R,
                                          N, H_q, H_kv, d, d_I, Bk, blk.shape[2], float(scale), float(kl_weight),
                                          _p(dq), _p(dqi), _p(kl), n_threads or threads())
    _check(rc, "msa_ref_sparse_attn_bwd_rows")
    return {"dq": dq, "dq_idx": dqi, "kl": kl}


def warmup_index(q, k, q_idx, k_idx, scale, kl_weight=1.0, rows=None, n_threads=None):
    """Warmup mode's index branch ("MSA" study note 4-4 "Indexer warmup"): the full-context teacher (mean over
    the group's heads of dense causal attention probabilities), the KL of each row and its gradients on q^I
    and k^I.  Returns dict(kl [G, R], dq_idx [R, G, d_I], dk_idx [N, d_I] or None with rows, lse_idx [G, R])."""
    q, k, q_idx, k_idx = _u16(q), _u16(k), _u16(q_idx), _u16(k_idx)
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    G, d_I = q_idx.shape[1], q_idx.shape[2]
    rr = None if rows is None else _i64(rows)
    R = N if rr is None else len(rr)
    kl = np.empty((G, R), np.float64)
    dq_idx = np.empty((R, G, d_I), np.float64)
    dk_idx = np.empty((N, d_I), np.float64) if rr is None else None
    lse_idx = np.empty((G, R), np.float64)
    _check(_load().msa_ref_warmup_index(_p(q), _p(k), _p(q_idx), _p(k_idx), _p(rr), R, N, H_q, H_kv, d, d_I,
                                        float(scale), float(kl_weight), _p(kl), _p(dq_idx), _p(dk_idx), _p(lse_idx),
                                        n_threads or threads()), "msa_ref_warmup_index")
    return dict(kl=kl, dq_idx=dq_idx, dk_idx=dk_idx, lse_idx=lse_idx)
