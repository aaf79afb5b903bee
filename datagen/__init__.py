"""Seeded synthetic inputs for the MSA forward path (test and benchmark infrastructure).

This module holds none of the method's arithmetic.  It generates the inputs
both sides consume: the fp64 CPU oracle (host arrays, any subset of rows) and
the CUDA path (device tensors filled in place).  Host and device fills share
``dg_core.h`` and agree bit for bit.

Recipe (the workloads of the pages: bf16 ~N(0,1) tensors plus planted
"needle" blocks whose index key is aligned with a random half of later index
queries):

* every tensor element is ``bf16(normal(seed, tensor_id, flat_index))``, a
  counter-based Irwin-Hall(8) approximation of N(0,1) (see ``dg_core.h``);
* per group ``g``, ``m`` needle blocks are drawn uniformly without replacement
  from the blocks that have later rows (prefill: ``b <= nb - 2``; decode:
  ``b < local(t)``), each with one needle token at a uniformly drawn offset;
* the ``G*m`` needle directions ``u`` are orthonormal (QR of a seeded Gaussian
  matrix, rounded to fp32);
* the needle token's index key is ``bf16(alpha * u)``, ``alpha = 4 sqrt(d_I)``;
* index-query row ``(t, g)`` picks each needle of its group whose block lies
  before ``local(t)`` with probability 1/2 (a seeded bit), capped at ``k - 1``
  picks, and becomes ``bf16(x + beta * sum(u_picked))`` with
  ``beta = 0.9 / sqrt(1 - 0.81) * sqrt(d_I)``, so that a single picked
  needle has cosine ~0.9 with the row.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libdg_host.so")
_CUDA_SO = os.path.join(_HERE, "libdg_cuda.so")

# tensor ids of the counter-based streams
TID = dict(q=1, k=2, v=3, q_idx=4, k_idx=5, pick=6,
           q_t=11, k_cache=12, v_cache=13, q_idx_t=14, k_idx_cache=15, pick_t=16,
           dout=21)

SEED_BASE = 0x4D5341


@dataclass
class Config:
    name: str
    kind: str  # "prefill" or "decode"
    H_q: int
    H_kv: int
    d: int
    d_I: int
    Bk: int
    k: int
    needles: int
    N: int = 0          # prefill tokens
    B: int = 0          # decode sequences
    ctx: int = 0        # decode cache length per sequence
    index: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def G(self):
        return self.H_kv

    @property
    def gs(self):
        return self.H_q // self.H_kv

    @property
    def nb(self):
        n = self.N if self.kind == "prefill" else self.ctx
        return (n + self.Bk - 1) // self.Bk

    @property
    def seed(self):
        return SEED_BASE + self.index


CONFIGS = {
    "tiny": Config("tiny", "prefill", N=1024, H_q=4, H_kv=1, d=64, d_I=32, Bk=64, k=4, needles=2, index=0),
    "prefill_32k": Config("prefill_32k", "prefill", N=32768, H_q=32, H_kv=8, d=128, d_I=128, Bk=128, k=16,
                          needles=4, index=1),
    "prefill_128k": Config("prefill_128k", "prefill", N=131072, H_q=64, H_kv=8, d=128, d_I=128, Bk=128,
                           k=16, needles=8, index=2),
    "decode_1m": Config("decode_1m", "decode", B=4, ctx=1 << 20, H_q=64, H_kv=8, d=128, d_I=128, Bk=128,
                        k=16, needles=4, index=3),
    # a smaller decode case (same shapes, 256K context) for profiler captures of a few GB
    "decode_256k": Config("decode_256k", "decode", B=4, ctx=1 << 18, H_q=64, H_kv=8, d=128, d_I=128, Bk=128,
                          k=16, needles=4, index=5),
    # a smaller prefill case (same shapes, N = 8K) for profiler captures of a few GB
    "prefill_8k": Config("prefill_8k", "prefill", N=8192, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=16,
                         needles=4, index=6),
    # the 128K shapes at N = 16K: q (268 MB) is larger than L2 while the attention call holds ~5 GB, so a
    # profiler capture of it sees DRAM traffic that scales with N to the 128K workload
    "prefill_16k": Config("prefill_16k", "prefill", N=16384, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=16,
                          needles=4, index=8),
    # the 32K head layout (gs = 4) at N = 16K: q (134 MB) is larger than L2 and the call holds ~2.5 GB
    "prefill_16k_gs4": Config("prefill_16k_gs4", "prefill", N=16384, H_q=32, H_kv=8, d=128, d_I=128, Bk=128,
                              k=16, needles=4, index=9),
    "prefill_1m": Config("prefill_1m", "prefill", N=1 << 20, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=16,
                         needles=16, index=4),
}


def make_config(name="custom", kind="prefill", index=100, **kw):
    return Config(name, kind, index=index, **kw)


# --------------------------------------------------------------------------- build / load
def build(verbose=False):
    """Compile the host (gcc) and device (nvcc) fill libraries in place."""
    src_h = os.path.join(_HERE, "dg_host.c")
    src_c = os.path.join(_HERE, "dg_cuda.cu")
    cmds = [
        ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-o", _HOST_SO, src_h],
        ["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-gencode", "arch=compute_103a,code=sm_103a",
         "-o", _CUDA_SO, src_c],
    ]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in cmds]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("datagen build failed: %s\n%s" % (" ".join(c), out.decode()))
        if verbose and out:
            print(out.decode())


_host_lib = None
_cuda_lib = None


def _host():
    global _host_lib
    if _host_lib is None:
        if not os.path.exists(_HOST_SO):
            build()
        lib = ctypes.CDLL(_HOST_SO)
        P, I64, U64, U32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        lib.dg_host_fill_normal.argtypes = [P, I64, U64, U32, I64, I]
        lib.dg_host_fill_normal_rows.argtypes = [P, P, I64, I64, U64, U32, I]
        lib.dg_host_q_idx_rows.argtypes = [P, P, P, I64, U64, U32, U32, I, I, I, I, I, P, P, ctypes.c_float, I]
        lib.dg_host_pick_masks.argtypes = [P, P, P, I64, U64, U32, I, I, I, I, P]
        _host_lib = lib
    return _host_lib


def _cuda():
    global _cuda_lib
    if _cuda_lib is None:
        if not os.path.exists(_CUDA_SO):
            raise RuntimeError("datagen CUDA library missing: run datagen.build()")
        lib = ctypes.CDLL(_CUDA_SO)
        P, I64, U64, U32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        lib.dg_cuda_fill_normal.argtypes = [P, I64, U64, U32, I64, P]
        lib.dg_cuda_fill_normal.restype = I
        lib.dg_cuda_q_idx.argtypes = [P, I64, P, U64, U32, U32, I, I, I, I, I, P, P, ctypes.c_float, P]
        lib.dg_cuda_q_idx.restype = I
        _cuda_lib = lib
    return _cuda_lib


def _threads():
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


# --------------------------------------------------------------------------- bf16 helpers
def bf16_to_f64(a_u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (a_u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (non-NaN inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return ((b >> 16) & 0xFFFF).astype(np.uint16)


# --------------------------------------------------------------------------- needles
@dataclass
class Needles:
    m: int
    cap: int
    blocks: np.ndarray   # [S, G, m] int32 (S = 1 for prefill, B for decode)
    offsets: np.ndarray  # [S, G, m] int32
    u: np.ndarray        # [G*m, d_I] float32, orthonormal rows
    alpha: np.float32
    beta: np.float32

    def tokens(self, Bk, s=0):
        return (self.blocks[s].astype(np.int64) * Bk + self.offsets[s]).reshape(-1)


def make_needles(cfg: Config, ctx_len=None) -> Needles:
    """Needle blocks, offsets and directions for a config (see module doc)."""
    G, m, d_I, Bk = cfg.G, cfg.needles, cfg.d_I, cfg.Bk
    rng = np.random.default_rng([cfg.seed, 0xA11CE])
    assert G * m <= d_I, "needle directions must fit in d_I"
    if m > 0:
        qmat, _ = np.linalg.qr(rng.standard_normal((d_I, G * m)))
        u = np.ascontiguousarray(qmat.T.astype(np.float32))
    else:
        u = np.zeros((0, d_I), np.float32)
    if cfg.kind == "prefill":
        limits = [cfg.nb - 1]  # blocks 0 .. nb-2 have later rows
    else:
        ctx_len = np.asarray(ctx_len if ctx_len is not None else [cfg.ctx] * cfg.B, np.int64)
        limits = [int((c - 1) // Bk) for c in ctx_len]  # blocks before the query's local block
    S = len(limits)
    blocks = np.full((S, G, m), -1, np.int32)
    offsets = np.zeros((S, G, m), np.int32)
    for s, lim in enumerate(limits):
        used = set()
        for g in range(G):
            if lim <= 0 or m == 0:
                continue
            take = min(m, lim)
            bl = rng.choice(lim, size=take, replace=False)
            for n in range(take):
                b = int(bl[n])
                while True:
                    o = int(rng.integers(0, Bk))
                    if (b, o) not in used:
                        used.add((b, o))
                        break
                blocks[s, g, n] = b
                offsets[s, g, n] = o
    alpha = np.float32(4.0 * math.sqrt(d_I))
    beta = np.float32(0.9 / math.sqrt(1.0 - 0.81) * math.sqrt(d_I))
    return Needles(m=m, cap=max(cfg.k - 1, 0), blocks=blocks, offsets=offsets, u=u, alpha=alpha, beta=beta)


def needle_key_rows(nd: Needles, s=0):
    """bf16 index-key rows of the needle tokens of sequence s: [G*m, d_I] uint16 (-1 blocks skipped)."""
    prod = (nd.alpha * nd.u).astype(np.float32)  # one fp32 rounding per element
    rows = f32_to_bf16_rne(prod)
    valid = nd.blocks[s].reshape(-1) >= 0
    return rows, valid


# --------------------------------------------------------------------------- host generation
def host_normal(n, seed, tid, first=0):
    out = np.empty(n, np.uint16)
    _host().dg_host_fill_normal(_ptr(out), n, seed, tid, first, _threads())
    return out


def host_normal_rows(row_ids, row_len, seed, tid):
    row_ids = np.ascontiguousarray(row_ids, np.int64)
    out = np.empty((len(row_ids), row_len), np.uint16)
    _host().dg_host_fill_normal_rows(_ptr(out), _ptr(row_ids), len(row_ids), row_len, seed, tid, _threads())
    return out


def host_q_idx_rows(cfg: Config, nd: Needles, row_ids, pos, noise_tid, pick_tid, s=0):
    row_ids = np.ascontiguousarray(row_ids, np.int64)
    pos = np.ascontiguousarray(pos, np.int64)
    out = np.empty((len(row_ids), cfg.G, cfg.d_I), np.uint16)
    nb_arr = np.ascontiguousarray(nd.blocks[s].reshape(-1), np.int32)
    _host().dg_host_q_idx_rows(_ptr(out), _ptr(row_ids), _ptr(pos), len(row_ids), cfg.seed, noise_tid, pick_tid,
                               cfg.G, cfg.d_I, cfg.Bk, nd.m, nd.cap, _ptr(nb_arr), _ptr(nd.u),
                               ctypes.c_float(nd.beta), _threads())
    return out


def pick_masks(cfg: Config, nd: Needles, row_ids, pos, pick_tid, s=0):
    """[n_rows, G] uint32: bit n set when index-query row (row_ids[i], position pos[i]) picked needle n."""
    row_ids = np.ascontiguousarray(row_ids, np.int64)
    pos = np.ascontiguousarray(pos, np.int64)
    out = np.empty((len(row_ids), cfg.G), np.uint32)
    nb_arr = np.ascontiguousarray(nd.blocks[s].reshape(-1), np.int32)
    _host().dg_host_pick_masks(_ptr(out), _ptr(row_ids), _ptr(pos), len(row_ids), cfg.seed, pick_tid, cfg.G, cfg.Bk,
                               nd.m, nd.cap, _ptr(nb_arr))
    return out


def prefill_host(cfg: Config, rows=None, want=("q", "k", "v", "q_idx", "k_idx")):
    """Host bf16 (uint16) prefill inputs.  With `rows`, q and q_idx hold only those positions."""
    N, H_q, H_kv, d, d_I, G = cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.G
    nd = make_needles(cfg)
    out = {"needles": nd}
    rows_arr = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    if "q" in want:
        if rows is None:
            out["q"] = host_normal(N * H_q * d, cfg.seed, TID["q"]).reshape(N, H_q, d)
        else:
            out["q"] = host_normal_rows(rows_arr, H_q * d, cfg.seed, TID["q"]).reshape(-1, H_q, d)
    if "k" in want:
        out["k"] = host_normal(N * H_kv * d, cfg.seed, TID["k"]).reshape(N, H_kv, d)
    if "v" in want:
        out["v"] = host_normal(N * H_kv * d, cfg.seed, TID["v"]).reshape(N, H_kv, d)
    if "q_idx" in want:
        out["q_idx"] = host_q_idx_rows(cfg, nd, rows_arr, rows_arr, TID["q_idx"], TID["pick"])
    if "k_idx" in want:
        ki = host_normal(N * d_I, cfg.seed, TID["k_idx"]).reshape(N, d_I)
        krows, valid = needle_key_rows(nd)
        toks = nd.tokens(cfg.Bk)
        ki[toks[valid]] = krows[valid]
        out["k_idx"] = ki
    return out


def decode_host(cfg: Config, ctx_len=None, want=("q_t", "q_idx_t", "k_idx_cache", "k_cache", "v_cache"),
                kv_tokens=None):
    """Host bf16 decode inputs.  `kv_tokens` (list per sequence of token arrays) limits the K/V
    caches to those tokens: the result then maps (b, token) -> row in dicts 'k_rows'/'v_rows'."""
    B, C, H_q, H_kv, d, d_I, G = cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.G
    ctx_len = np.asarray(ctx_len if ctx_len is not None else [C] * B, np.int64)
    nd = make_needles(cfg, ctx_len)
    out = {"needles": nd, "ctx_len": ctx_len}
    if "q_t" in want:
        out["q_t"] = host_normal(B * H_q * d, cfg.seed, TID["q_t"]).reshape(B, H_q, d)
    if "q_idx_t" in want:
        qi = np.empty((B, G, d_I), np.uint16)
        for b in range(B):
            qi[b] = host_q_idx_rows(cfg, nd, [b], [ctx_len[b] - 1], TID["q_idx_t"], TID["pick_t"], s=b)[0]
        out["q_idx_t"] = qi
    if "k_idx_cache" in want:
        ki = host_normal(B * C * d_I, cfg.seed, TID["k_idx_cache"]).reshape(B, C, d_I)
        for b in range(B):
            krows, valid = needle_key_rows(nd, b)
            toks = nd.tokens(cfg.Bk, b)
            ki[b, toks[valid]] = krows[valid]
        out["k_idx_cache"] = ki
    for name in ("k_cache", "v_cache"):
        if name not in want:
            continue
        if kv_tokens is None:
            out[name] = host_normal(B * C * H_kv * d, cfg.seed, TID[name]).reshape(B, C, H_kv, d)
        else:
            rows = {}
            for b, toks in enumerate(kv_tokens):
                toks = np.asarray(toks, np.int64)
                ids = b * C + toks
                vals = host_normal_rows(ids, H_kv * d, cfg.seed, TID[name]).reshape(-1, H_kv, d)
                rows[b] = (toks, vals)
            out[name + "_rows"] = rows
    return out


# --------------------------------------------------------------------------- device generation
def device_normal_(t, seed, tid, first=0):
    """Fill a contiguous bf16 CUDA tensor in place with the normal stream."""
    import torch
    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    rc = _cuda().dg_cuda_fill_normal(ctypes.c_void_p(t.data_ptr()), t.numel(), seed, tid, first,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise RuntimeError("dg_cuda_fill_normal failed: %d" % rc)
    return t


def _u16_to_bf16_tensor(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def prefill_device(cfg: Config, device="cuda", want=("q", "k", "v", "q_idx", "k_idx")):
    """Device bf16 prefill inputs (q, k, v, q_idx, k_idx) filled in place on the GPU."""
    import torch
    N, H_q, H_kv, d, d_I, G = cfg.N, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.G
    nd = make_needles(cfg)
    bf = torch.bfloat16
    out = dict(needles=nd)
    for name, shp in (("q", (N, H_q, d)), ("k", (N, H_kv, d)), ("v", (N, H_kv, d))):
        if name in want:
            out[name] = device_normal_(torch.empty(shp, dtype=bf, device=device), cfg.seed, TID[name])
    if "k_idx" in want:
        k_idx = device_normal_(torch.empty((N, d_I), dtype=bf, device=device), cfg.seed, TID["k_idx"])
        krows, valid = needle_key_rows(nd)
        toks = nd.tokens(cfg.Bk)
        if valid.any():
            idx = torch.from_numpy(toks[valid]).to(device)
            k_idx[idx] = _u16_to_bf16_tensor(krows[valid]).to(device)
        out["k_idx"] = k_idx
    if "q_idx" in want:
        q_idx = torch.empty((N, G, d_I), dtype=bf, device=device)
        nb_dev = torch.from_numpy(np.ascontiguousarray(nd.blocks[0].reshape(-1), np.int32)).to(device)
        u_dev = torch.from_numpy(nd.u).to(device) if nd.u.size else torch.zeros(1, device=device)
        rc = _cuda().dg_cuda_q_idx(ctypes.c_void_p(q_idx.data_ptr()), N, None, cfg.seed, TID["q_idx"], TID["pick"],
                                   G, d_I, cfg.Bk, nd.m, nd.cap, ctypes.c_void_p(nb_dev.data_ptr()),
                                   ctypes.c_void_p(u_dev.data_ptr()), ctypes.c_float(nd.beta),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if rc != 0:
            raise RuntimeError("dg_cuda_q_idx failed: %d" % rc)
        out["q_idx"] = q_idx
    return out


def decode_device(cfg: Config, ctx_len=None, device="cuda"):
    """Device bf16 decode inputs; the small per-sequence query rows come from the host generator."""
    import torch
    B, C, H_q, H_kv, d, d_I, G = cfg.B, cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.G
    ctx_len = np.asarray(ctx_len if ctx_len is not None else [C] * B, np.int64)
    host = decode_host(cfg, ctx_len, want=("q_t", "q_idx_t"))
    nd = host["needles"]
    bf = torch.bfloat16
    k_idx_cache = device_normal_(torch.empty((B, C, d_I), dtype=bf, device=device), cfg.seed, TID["k_idx_cache"])
    for b in range(B):
        krows, valid = needle_key_rows(nd, b)
        toks = nd.tokens(cfg.Bk, b)
        if valid.any():
            idx = torch.from_numpy(toks[valid]).to(device)
            k_idx_cache[b, idx] = _u16_to_bf16_tensor(krows[valid]).to(device)
    k_cache = device_normal_(torch.empty((B, C, H_kv, d), dtype=bf, device=device), cfg.seed, TID["k_cache"])
    v_cache = device_normal_(torch.empty((B, C, H_kv, d), dtype=bf, device=device), cfg.seed, TID["v_cache"])
    return dict(q_t=_u16_to_bf16_tensor(host["q_t"]).to(device),
                q_idx_t=_u16_to_bf16_tensor(host["q_idx_t"]).to(device),
                k_idx_cache=k_idx_cache, k_cache=k_cache, v_cache=v_cache,
                ctx_len=torch.from_numpy(ctx_len.astype(np.int32)).to(device), ctx_len_host=ctx_len,
                needles=nd)


def to_bf16_tensor(a_u16):
    """Host uint16 bf16 bit patterns -> torch.bfloat16 CPU tensor (no copy)."""
    return _u16_to_bf16_tensor(a_u16)


def sample_rows(N, n, seed, must=()):
    """Seeded sample of n distinct positions in [0, N), always including `must` (sorted)."""
    rng = np.random.default_rng([seed, 0x5A3])
    must = [int(x) for x in must if 0 <= x < N]
    pool = np.setdiff1d(np.arange(N, dtype=np.int64), np.asarray(must, np.int64)) if N <= (1 << 22) else None
    n_rand = max(0, min(n, N) - len(must))
    if pool is not None:
        extra = rng.choice(pool, size=min(n_rand, len(pool)), replace=False)
    else:
        extra = set()
        while len(extra) < n_rand:
            x = int(rng.integers(0, N))
            if x not in must:
                extra.add(x)
        extra = np.fromiter(extra, np.int64)
    return np.unique(np.concatenate([np.asarray(must, np.int64), np.asarray(extra, np.int64)]))
