"""ctypes binding of libmsa.so: the C ABI of include/msa.h under the same names.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (bf16 as ``torch.bfloat16``, int32 as
``torch.int32``); their device pointers and the current torch stream are
passed through.  Importing this module loads ``libmsa.so`` and fails loudly if
it is missing — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libmsa.so is not built (run __graft_entry__.build() or "
                      "python -m block_sparse_long_index_gb300.build); there is no fallback path")
_lib = ctypes.CDLL(LIB_PATH)

MSA_OK = 0
MSA_ERR_INVALID_ARGUMENT = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_WORKSPACE_TOO_SMALL = 3
MSA_ERR_CUDA = 4
MSA_ERR_BAD_INDEX = 5
MSA_ERR_TIMEOUT = 6


class msa_shape_t(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int), ("d", ctypes.c_int),
                ("d_I", ctypes.c_int), ("Bk", ctypes.c_int), ("k", ctypes.c_int)]


_P, _I64, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_SP = ctypes.POINTER(msa_shape_t)

_SIGS = {
    "msa_select_blocks_workspace": (_SZ, [_I64, _I, _I, _I, _I]),
    "msa_select_blocks": (_I, [_P, _P, _I64, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "msa_invert_blocks_workspace": (_SZ, [_I64, _I, _I, _I]),
    "msa_invert_blocks": (_I, [_P, _I64, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "msa_sparse_attn_fwd_workspace": (_SZ, [_SP]),
    "msa_sparse_attn_fwd": (_I, [_P, _P, _P, _P, _SP, _F, _P, _P, _P, _SZ, _P]),
    "msa_sparse_attn_bwd_workspace": (_SZ, [_SP]),
    "msa_sparse_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SP, _F, _F, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                 _P]),
    "msa_prefill_workspace": (_SZ, [_SP]),
    "msa_prefill": (_I, [_P, _P, _P, _P, _P, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_decode_workspace": (_SZ, [_I, _SP]),
    "msa_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, _I, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _SP, _F, _P, _P, _P, _P]),
    "msa_quantize_e4m3": (_I, [_P, _I64, _F, _P, _P]),
    "msa_warmup_fwd": (_I, [_P, _P, _P, _P, _P, _SP, _F, _P, _P, _P, _P]),
    "msa_warmup_index_grad": (_I, [_P, _P, _P, _P, _P, _P, _SP, _F, _F, _P, _P, _P, _P]),
    "msa_select_blocks_varlen_workspace": (_SZ, [_I64, _I, _I, _I, _I]),
    "msa_select_blocks_varlen": (_I, [_P, _P, _P, _I, _I64, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "msa_prefill_varlen_workspace": (_SZ, [_SP]),
    "msa_prefill_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_select_blocks_fp8": (_I, [_P, _P, _I64, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "msa_prefill_fp8": (_I, [_P, _P, _P, _P, _P, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_decode_paged_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, _I, _SP, _F, _P, _P, _P, _P, _SZ, _P]),
    "msa_check_device_error": (_I, [_P, _P]),
    "msa_status_string": (ctypes.c_char_p, [_I]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTS = tuple(_SIGS)


class MsaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, msa_status_string(status), status))


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr() if hasattr(t, "data_ptr") else int(t))


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status, where):
    if status != MSA_OK:
        raise MsaError(status, where)
    return status


def shape(N, H_q, H_kv, d, d_I, Bk, k):
    return msa_shape_t(int(N), int(H_q), int(H_kv), int(d), int(d_I), int(Bk), int(k))


# ---------------------------------------------------------------- same-name wrappers
def msa_status_string(status):
    return _lib.msa_status_string(int(status)).decode()


def msa_select_blocks_workspace(N, G, d_I, Bk, k):
    return int(_lib.msa_select_blocks_workspace(N, G, d_I, Bk, k))


def msa_select_blocks(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_select_blocks(_ptr(q_idx), _ptr(k_idx), N, G, d_I, Bk, k, _ptr(block_idx),
                                         _ptr(workspace), wb, _stream(stream)), "msa_select_blocks")


def msa_invert_blocks_workspace(N, G, Bk, k):
    return int(_lib.msa_invert_blocks_workspace(N, G, Bk, k))


def msa_invert_blocks(block_idx, N, G, Bk, k, row_ptr, entries, n_entries, workspace, workspace_bytes=None,
                      stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_invert_blocks(_ptr(block_idx), N, G, Bk, k, _ptr(row_ptr), _ptr(entries),
                                         _ptr(n_entries), _ptr(workspace), wb, _stream(stream)),
                  "msa_invert_blocks")


def msa_sparse_attn_fwd_workspace(shp):
    return int(_lib.msa_sparse_attn_fwd_workspace(ctypes.byref(shp)))


def msa_sparse_attn_fwd(q, k, v, block_idx, shp, scale, out, lse, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_sparse_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(block_idx), ctypes.byref(shp),
                                           float(scale), _ptr(out), _ptr(lse), _ptr(workspace), wb,
                                           _stream(stream)), "msa_sparse_attn_fwd")


def msa_sparse_attn_bwd_workspace(shp):
    return int(_lib.msa_sparse_attn_bwd_workspace(ctypes.byref(shp)))


def msa_sparse_attn_bwd(q, k, v, q_idx, k_idx, block_idx, out, lse, dout, shp, scale, kl_weight, dq, dk, dv, dq_idx,
                        dk_idx, kl, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_sparse_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), _ptr(block_idx),
                                           _ptr(out), _ptr(lse), _ptr(dout), ctypes.byref(shp), float(scale),
                                           float(kl_weight), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dq_idx), _ptr(dk_idx),
                                           _ptr(kl), _ptr(workspace), wb, _stream(stream)), "msa_sparse_attn_bwd")


def msa_prefill_workspace(shp):
    return int(_lib.msa_prefill_workspace(ctypes.byref(shp)))


def msa_prefill(q, k, v, q_idx, k_idx, shp, scale, block_idx, out, lse, workspace, workspace_bytes=None,
                stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), ctypes.byref(shp),
                                   float(scale), _ptr(block_idx), _ptr(out), _ptr(lse), _ptr(workspace), wb,
                                   _stream(stream)), "msa_prefill")


def msa_decode_workspace(B, shp):
    return int(_lib.msa_decode_workspace(B, ctypes.byref(shp)))


def msa_decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, B, shp, scale, out, lse, block_idx,
               workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_decode(_ptr(q_t), _ptr(q_idx_t), _ptr(k_idx_cache), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(ctx_len), B, ctypes.byref(shp), float(scale), _ptr(out), _ptr(lse),
                                  _ptr(block_idx), _ptr(workspace), wb, _stream(stream)), "msa_decode")


def msa_decode_paged(q_t, q_idx_t, k_idx_pool, k_pool, v_pool, page_table, max_pages, n_pages, page_size, ctx_len,
                     B, shp, scale, out, lse, block_idx, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_decode_paged(_ptr(q_t), _ptr(q_idx_t), _ptr(k_idx_pool), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(page_table), int(max_pages), int(n_pages), int(page_size), _ptr(ctx_len),
                                        B, ctypes.byref(shp), float(scale), _ptr(out), _ptr(lse), _ptr(block_idx),
                                        _ptr(workspace), wb, _stream(stream)), "msa_decode_paged")


def msa_decode_noalloc(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, B, shp, scale, out, lse, block_idx,
                       stream=None):
    """msa_decode without a workspace, for callers that may not allocate device memory (the library's
    fixed 8 MiB device array is the scratch; calls on one device must not overlap)."""
    return _check(_lib.msa_decode_noalloc(_ptr(q_t), _ptr(q_idx_t), _ptr(k_idx_cache), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(ctx_len), B, ctypes.byref(shp), float(scale), _ptr(out), _ptr(lse),
                                          _ptr(block_idx), _stream(stream)), "msa_decode_noalloc")


def msa_quantize_e4m3(x, n, scale, y, stream=None):
    return _check(_lib.msa_quantize_e4m3(_ptr(x), int(n), float(scale), _ptr(y), _stream(stream)),
                  "msa_quantize_e4m3")


def msa_select_blocks_fp8(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_select_blocks_fp8(_ptr(q_idx), _ptr(k_idx), N, G, d_I, Bk, k, _ptr(block_idx),
                                             _ptr(workspace), wb, _stream(stream)), "msa_select_blocks_fp8")


def msa_prefill_fp8(q, k, v, q_idx, k_idx, shp, scale, block_idx, out, lse, workspace, workspace_bytes=None,
                    stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_prefill_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), ctypes.byref(shp),
                                       float(scale), _ptr(block_idx), _ptr(out), _ptr(lse), _ptr(workspace), wb,
                                       _stream(stream)), "msa_prefill_fp8")


def msa_decode_fp8(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, B, shp, scale, out, lse, block_idx,
                   workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_decode_fp8(_ptr(q_t), _ptr(q_idx_t), _ptr(k_idx_cache), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(ctx_len), B, ctypes.byref(shp), float(scale), _ptr(out), _ptr(lse),
                                      _ptr(block_idx), _ptr(workspace), wb, _stream(stream)), "msa_decode_fp8")


def msa_decode_paged_fp8(q_t, q_idx_t, k_idx_pool, k_pool, v_pool, page_table, max_pages, n_pages, page_size,
                         ctx_len, B, shp, scale, out, lse, block_idx, workspace, workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_decode_paged_fp8(_ptr(q_t), _ptr(q_idx_t), _ptr(k_idx_pool), _ptr(k_pool),
                                            _ptr(v_pool), _ptr(page_table), int(max_pages), int(n_pages),
                                            int(page_size), _ptr(ctx_len), B, ctypes.byref(shp), float(scale),
                                            _ptr(out), _ptr(lse), _ptr(block_idx), _ptr(workspace), wb,
                                            _stream(stream)), "msa_decode_paged_fp8")


def msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k):
    return int(_lib.msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k))


def msa_select_blocks_varlen(q_idx, k_idx, cu_seqlens, S, N, G, d_I, Bk, k, block_idx, workspace,
                             workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_select_blocks_varlen(_ptr(q_idx), _ptr(k_idx), _ptr(cu_seqlens), int(S), N, G, d_I, Bk,
                                                k, _ptr(block_idx), _ptr(workspace), wb, _stream(stream)),
                  "msa_select_blocks_varlen")


def msa_prefill_varlen_workspace(shp):
    return int(_lib.msa_prefill_varlen_workspace(ctypes.byref(shp)))


def msa_prefill_varlen(q, k, v, q_idx, k_idx, cu_seqlens, S, shp, scale, block_idx, out, lse, workspace,
                       workspace_bytes=None, stream=None):
    wb = workspace.numel() if workspace_bytes is None else workspace_bytes
    return _check(_lib.msa_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), _ptr(cu_seqlens),
                                          int(S), ctypes.byref(shp), float(scale), _ptr(block_idx), _ptr(out),
                                          _ptr(lse), _ptr(workspace), wb, _stream(stream)), "msa_prefill_varlen")


def msa_warmup_fwd(q, k, v, q_idx, k_idx, shp, scale, out, lse, lse_idx, stream=None):
    return _check(_lib.msa_warmup_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), ctypes.byref(shp),
                                      float(scale), _ptr(out), _ptr(lse), _ptr(lse_idx), _stream(stream)),
                  "msa_warmup_fwd")


def msa_warmup_index_grad(q, k, q_idx, k_idx, lse, lse_idx, shp, scale, kl_weight, dq_idx, dk_idx, kl, stream=None):
    return _check(_lib.msa_warmup_index_grad(_ptr(q), _ptr(k), _ptr(q_idx), _ptr(k_idx), _ptr(lse), _ptr(lse_idx),
                                             ctypes.byref(shp), float(scale), float(kl_weight), _ptr(dq_idx),
                                             _ptr(dk_idx), _ptr(kl), _stream(stream)), "msa_warmup_index_grad")


def msa_check_device_error(workspace, stream=None):
    """Returns the device status code (raises nothing)."""
    return int(_lib.msa_check_device_error(_ptr(workspace), _stream(stream)))


def raw():
    """The loaded ctypes library (for status-code tests that bypass the wrappers)."""
    return _lib
