"""INT4 per-(token, head) KV cache for NVIDIA GB300: Python binding of the C ABI in include/kv_int4.h.

The functions below have the C entry points' names.  They only marshal arguments: check that the
torch tensors are CUDA, contiguous and of the right dtype and shape, then pass raw device pointers
and the current CUDA stream to ``libkv_int4.so``.  Every step of the write and of the attention
runs in that library's kernels; there is no fallback: the first call (or ``load()``) raises
ImportError when the library has not been built (``python int4_token_head_kv_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkv_int4.so")

KV_INT4_F16, KV_INT4_BF16, KV_INT4_F32 = 0, 1, 2
STAT_NAMES = ["slot_out_of_range", "block_out_of_range", "bad_sequence", "wait_timeout", "bad_sign"]
_STAT_COUNT = 8
_DTYPES = {torch.float16: KV_INT4_F16, torch.bfloat16: KV_INT4_BF16, torch.float32: KV_INT4_F32}


class AttnOptions(ctypes.Structure):
    """kv_int4_attn_options: window_left (< 0: none), softcap (0: none), alibi_slopes (device
    pointer to fp32 [num_q_heads], or None), qq_bias (device pointer to fp32 rows of
    qq_bias_stride elements, or None)."""
    _fields_ = [("window_left", ctypes.c_int32), ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("qq_bias", ctypes.c_void_p), ("qq_bias_stride", ctypes.c_int32)]


class KVInt4Error(RuntimeError):
    """A non-OK status returned by the C library."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m int4_token_head_kv_gb300._build` "
                          "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, szt = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kv_int4_row_bytes.argtypes = [i32]
    lib.kv_int4_row_bytes.restype = i32
    lib.kv_int4_status_string.argtypes = [ctypes.c_int]
    lib.kv_int4_status_string.restype = ctypes.c_char_p
    lib.kv_int4_write.argtypes = [vp, vp, ctypes.c_int, i64, i32, i32, vp, vp, vp, i64, i32, vp]
    lib.kv_int4_write.restype = ctypes.c_int
    lib.kv_int8_row_bytes.argtypes = [i32]
    lib.kv_int8_row_bytes.restype = i32
    lib.kv_int8_write.argtypes = [vp, vp, ctypes.c_int, i64, i32, i32, vp, vp, i64, i32, vp]
    lib.kv_int8_write.restype = ctypes.c_int
    lib.kv_int2_row_bytes.argtypes = [i32]
    lib.kv_int2_row_bytes.restype = i32
    lib.kv_int2_write.argtypes = lib.kv_int4_write.argtypes
    lib.kv_int2_write.restype = ctypes.c_int
    lib.kv_int4_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.kv_int4_attention_workspace_bytes.restype = szt
    lib.kv_int4_attention_segment_len.argtypes = [i32, i32, i32]
    lib.kv_int4_attention_segment_len.restype = i32
    lib.kv_int4_paged_attention.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp,
                                            i32, i32, i32, f32, vp, i32, vp, ctypes.c_int, vp, szt, vp]
    lib.kv_int4_paged_attention.restype = ctypes.c_int
    lib.kv_int4_paged_attention_noalloc.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp,
                                                    vp, i32, i32, i32, f32, vp, i32, vp, ctypes.c_int, vp]
    lib.kv_int4_paged_attention_noalloc.restype = ctypes.c_int
    lib.kv_int4_paged_attention_noalloc_ex.argtypes = lib.kv_int4_paged_attention_noalloc.argtypes + [
        ctypes.POINTER(AttnOptions)]
    lib.kv_int4_paged_attention_noalloc_ex.restype = ctypes.c_int
    lib.kv_int4_paged_attention_ex.argtypes = lib.kv_int4_paged_attention.argtypes + [ctypes.POINTER(AttnOptions)]
    lib.kv_int4_paged_attention_ex.restype = ctypes.c_int
    lib.kv_int8_paged_attention.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp,
                                            i32, i32, i32, f32, i32, vp, ctypes.c_int, vp, szt, vp]
    lib.kv_int8_paged_attention.restype = ctypes.c_int
    lib.kv_int2_paged_attention.argtypes = lib.kv_int4_paged_attention.argtypes
    lib.kv_int2_paged_attention.restype = ctypes.c_int
    lib.kv_int4_read_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.kv_int4_read_device_status.restype = ctypes.c_int
    lib.kv_int4_clear_device_status.argtypes = [vp]
    lib.kv_int4_clear_device_status.restype = ctypes.c_int
    lib.kv_int4_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.kv_int4_selftest_wait_timeout.restype = ctypes.c_int
    return lib


_lib = None


def load():
    """Load libkv_int4.so (once); raises ImportError when it has not been built."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise KVInt4Error(fn, status, load().kv_int4_status_string(status).decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _one_device(*tensors) -> torch.device:
    """The device all the given CUDA tensors (None entries skipped) are on; the library launches on the
    current device, so the calls below make it this one."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def _cuda(t: torch.Tensor, name: str, dtypes=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t


def kv_int4_row_bytes(head_size: int) -> int:
    return int(load().kv_int4_row_bytes(head_size))


def kv_int4_cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    """Shape of the packed cache: (num_blocks, 2, block_size, num_kv_heads, head_size/2 + 4) uint8."""
    return (num_blocks, 2, block_size, num_kv_heads, kv_int4_row_bytes(head_size))


def kv_int4_write(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor, rht_signs: torch.Tensor,
                  kv_cache: torch.Tensor, stream=None) -> None:
    """Rotate, quantise and pack ``key``/``value`` [T, H, d] into ``kv_cache`` at ``slot_mapping``."""
    _rotated_write("kv_int4_write", kv_int4_row_bytes, key, value, slot_mapping, rht_signs, kv_cache, stream)


def _rotated_write(fn, row_bytes, key, value, slot_mapping, rht_signs, kv_cache, stream):
    _cuda(key, "key", (torch.float16, torch.bfloat16))
    _cuda(value, "value", (key.dtype,))
    _cuda(slot_mapping, "slot_mapping", (torch.int64,))
    _cuda(rht_signs, "rht_signs", (torch.float32,))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key and value must both be [num_tokens, num_kv_heads, head_size]")
    T, H, d = key.shape
    if slot_mapping.shape != (T,) or rht_signs.shape != (d,):
        raise ValueError("slot_mapping must be [num_tokens] and rht_signs [head_size]")
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2 or kv_cache.shape[3] != H or \
            kv_cache.shape[4] != row_bytes(d):
        raise ValueError(f"kv_cache must be (NB, 2, bs, {H}, {row_bytes(d)})")
    with torch.cuda.device(_one_device(key, value, slot_mapping, rht_signs, kv_cache)):
        st = getattr(load(), fn)(key.data_ptr(), value.data_ptr(), _DTYPES[key.dtype], T, H, d,
                                 slot_mapping.data_ptr(), rht_signs.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0],
                                 kv_cache.shape[2], _stream(stream))
    _check(fn, st)


def kv_int8_row_bytes(head_size: int) -> int:
    return int(load().kv_int8_row_bytes(head_size))


def kv_int8_cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    """INT8 per-(token, head) comparator cache: (num_blocks, 2, block_size, H, head_size + 4) uint8."""
    return (num_blocks, 2, block_size, num_kv_heads, kv_int8_row_bytes(head_size))


def kv_int8_write(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor, kv_cache: torch.Tensor,
                  stream=None) -> None:
    """Quantise ``key``/``value`` [T, H, d] to INT8 per-(token, head) rows of ``kv_cache`` at ``slot_mapping``."""
    _cuda(key, "key", (torch.float16, torch.bfloat16))
    _cuda(value, "value", (key.dtype,))
    _cuda(slot_mapping, "slot_mapping", (torch.int64,))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key and value must both be [num_tokens, num_kv_heads, head_size]")
    T, H, d = key.shape
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2 or kv_cache.shape[3] != H or \
            kv_cache.shape[4] != kv_int8_row_bytes(d):
        raise ValueError(f"kv_cache must be {kv_int8_cache_shape('NB', 'bs', H, d)}")
    with torch.cuda.device(_one_device(key, value, slot_mapping, kv_cache)):
        st = load().kv_int8_write(key.data_ptr(), value.data_ptr(), _DTYPES[key.dtype], T, H, d,
                                  slot_mapping.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0], kv_cache.shape[2],
                                  _stream(stream))
    _check("kv_int8_write", st)


def kv_int2_row_bytes(head_size: int) -> int:
    return int(load().kv_int2_row_bytes(head_size))


def kv_int2_cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    """INT2 Lloyd-Max cache: (num_blocks, 2, block_size, H, head_size/4 + 4) uint8."""
    return (num_blocks, 2, block_size, num_kv_heads, kv_int2_row_bytes(head_size))


def kv_int2_write(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor, rht_signs: torch.Tensor,
                  kv_cache: torch.Tensor, stream=None) -> None:
    """Rotate ``key``/``value`` [T, H, d] as kv_int4_write does, quantise them to INT2 Lloyd-Max codes
    and pack them into ``kv_cache`` at ``slot_mapping``."""
    _rotated_write("kv_int2_write", kv_int2_row_bytes, key, value, slot_mapping, rht_signs, kv_cache, stream)


def kv_int4_attention_segment_len(num_seqs: int, max_seq_len: int, segment_len: int = 0) -> int:
    return int(load().kv_int4_attention_segment_len(num_seqs, max_seq_len, segment_len))


def kv_int4_attention_workspace_bytes(num_q_heads: int, num_kv_heads: int, head_size: int, num_seqs: int,
                                      max_seq_len: int, segment_len: int = 0) -> int:
    return int(load().kv_int4_attention_workspace_bytes(num_q_heads, num_kv_heads, head_size, num_seqs,
                                                      max_seq_len, segment_len))


def _options(Hq, max_query_len, window_left, softcap, alibi_slopes, qq_bias):
    """kv_int4_attn_options for the given keywords, or None when none is set."""
    if window_left < 0 and softcap == 0.0 and alibi_slopes is None and qq_bias is None:
        return None
    if alibi_slopes is not None:
        _cuda(alibi_slopes, "alibi_slopes", (torch.float32,))
        if alibi_slopes.shape != (Hq,):
            raise ValueError("alibi_slopes must be [num_q_heads]")
    if qq_bias is not None:
        _cuda(qq_bias, "qq_bias", (torch.float32,))
        if qq_bias.dim() != 2 or qq_bias.stride(1) != 1 or qq_bias.shape[0] < max_query_len:
            raise ValueError("qq_bias must be a row-contiguous [rows >= max_query_len, cols] matrix")
    return AttnOptions(int(window_left), float(softcap),
                       alibi_slopes.data_ptr() if alibi_slopes is not None else None,
                       qq_bias.data_ptr() if qq_bias is not None else None,
                       int(qq_bias.stride(0)) if qq_bias is not None else 0)


def kv_int4_paged_attention(query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                            seq_lens: torch.Tensor, query_start_loc: torch.Tensor, softmax_scale: float,
                            rht_signs: torch.Tensor, max_query_len: int, max_seq_len: int, out=None,
                            out_dtype=None, segment_len: int = 0, workspace=None, stream=None,
                            window_left: int = -1, softcap: float = 0.0, alibi_slopes=None,
                            qq_bias=None) -> torch.Tensor:
    """Causal paged attention of ``query`` [Nq, Hq, d] over the INT4 cache; returns ``out``.  With
    ``window_left >= 0``, ``softcap > 0``, ``alibi_slopes`` (fp32 [Hq] on the device) or ``qq_bias``
    (fp32 [rows >= max_query_len, stride >= max_query_len] on the device, contiguous rows) the call
    goes through kv_int4_paged_attention_ex."""
    _cuda(query, "query", (torch.float16, torch.bfloat16))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    _cuda(block_tables, "block_tables", (torch.int32,))
    _cuda(seq_lens, "seq_lens", (torch.int32,))
    _cuda(query_start_loc, "query_start_loc", (torch.int32,))
    _cuda(rht_signs, "rht_signs", (torch.float32,))
    Nq, Hq, d = query.shape
    NB, two, bs, H, rb = kv_cache.shape
    S = seq_lens.shape[0]
    if two != 2 or rb != kv_int4_row_bytes(d) or rht_signs.shape != (d,):
        raise ValueError("kv_cache / rht_signs do not match the query's head size")
    if query_start_loc.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks] and query_start_loc [num_seqs + 1]")
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=out_dtype or query.dtype, device=query.device)
    _cuda(out, "out", tuple(_DTYPES))
    if out.shape != query.shape:
        raise ValueError("out must have the query's shape")
    need = kv_int4_attention_workspace_bytes(Hq, H, d, S, max_seq_len, segment_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = _options(Hq, max_query_len, window_left, softcap, alibi_slopes, qq_bias)
    with torch.cuda.device(_one_device(query, kv_cache, block_tables, seq_lens, query_start_loc, rht_signs, out,
                                       workspace, alibi_slopes, qq_bias)):
        args = (query.data_ptr(), _DTYPES[query.dtype], Nq, Hq, kv_cache.data_ptr(), NB, H, d, bs,
                block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), S,
                max_query_len, max_seq_len, float(softmax_scale), rht_signs.data_ptr(), segment_len, out.data_ptr(),
                _DTYPES[out.dtype], ws_ptr, ws_bytes, _stream(stream))
        if opts is not None:
            st, fn = load().kv_int4_paged_attention_ex(*args, ctypes.byref(opts)), "kv_int4_paged_attention_ex"
        else:
            st, fn = load().kv_int4_paged_attention(*args), "kv_int4_paged_attention"
    _check(fn, st)
    return out


def kv_int4_paged_attention_noalloc(query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                                    seq_lens: torch.Tensor, query_start_loc: torch.Tensor, softmax_scale: float,
                                    rht_signs: torch.Tensor, max_query_len: int, max_seq_len: int, out=None,
                                    out_dtype=None, segment_len: int = 0, stream=None, window_left: int = -1,
                                    softcap: float = 0.0, alibi_slopes=None, qq_bias=None) -> torch.Tensor:
    """kv_int4_paged_attention without a workspace: the split-KV partials live in the library's fixed
    device scratch array (calls that overlap on the GPU must be serialised).  ``out`` is allocated
    here when not given; pass it to keep the call free of allocations.  The options as for
    kv_int4_paged_attention (through kv_int4_paged_attention_noalloc_ex)."""
    _cuda(query, "query", (torch.float16, torch.bfloat16))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    _cuda(block_tables, "block_tables", (torch.int32,))
    _cuda(seq_lens, "seq_lens", (torch.int32,))
    _cuda(query_start_loc, "query_start_loc", (torch.int32,))
    _cuda(rht_signs, "rht_signs", (torch.float32,))
    Nq, Hq, d = query.shape
    NB, two, bs, H, rb = kv_cache.shape
    S = seq_lens.shape[0]
    if two != 2 or rb != kv_int4_row_bytes(d) or rht_signs.shape != (d,):
        raise ValueError("kv_cache / rht_signs do not match the query's head size")
    if query_start_loc.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks] and query_start_loc [num_seqs + 1]")
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=out_dtype or query.dtype, device=query.device)
    _cuda(out, "out", tuple(_DTYPES))
    if out.shape != query.shape:
        raise ValueError("out must have the query's shape")
    opts = _options(Hq, max_query_len, window_left, softcap, alibi_slopes, qq_bias)
    with torch.cuda.device(_one_device(query, kv_cache, block_tables, seq_lens, query_start_loc, rht_signs, out,
                                       alibi_slopes, qq_bias)):
        args = (query.data_ptr(), _DTYPES[query.dtype], Nq, Hq, kv_cache.data_ptr(), NB, H, d, bs,
                block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), S,
                max_query_len, max_seq_len, float(softmax_scale), rht_signs.data_ptr(), segment_len, out.data_ptr(),
                _DTYPES[out.dtype], _stream(stream))
        if opts is None:
            st, fn = load().kv_int4_paged_attention_noalloc(*args), "kv_int4_paged_attention_noalloc"
        else:
            st, fn = (load().kv_int4_paged_attention_noalloc_ex(*args, ctypes.byref(opts)),
                      "kv_int4_paged_attention_noalloc_ex")
    _check(fn, st)
    return out


def kv_int8_paged_attention(query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                            seq_lens: torch.Tensor, query_start_loc: torch.Tensor, softmax_scale: float,
                            max_query_len: int, max_seq_len: int, out=None, out_dtype=None, segment_len: int = 0,
                            workspace=None, stream=None) -> torch.Tensor:
    """Decode attention of ``query`` [Nq, Hq, d] (one query token per sequence) over the INT8
    comparator's cache; returns ``out``.  The workspace size is the INT4 call's."""
    _cuda(query, "query", (torch.float16, torch.bfloat16))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    _cuda(block_tables, "block_tables", (torch.int32,))
    _cuda(seq_lens, "seq_lens", (torch.int32,))
    _cuda(query_start_loc, "query_start_loc", (torch.int32,))
    Nq, Hq, d = query.shape
    NB, two, bs, H, rb = kv_cache.shape
    S = seq_lens.shape[0]
    if two != 2 or rb != kv_int8_row_bytes(d):
        raise ValueError("kv_cache does not match the query's head size")
    if query_start_loc.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks] and query_start_loc [num_seqs + 1]")
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=out_dtype or query.dtype, device=query.device)
    _cuda(out, "out", tuple(_DTYPES))
    if out.shape != query.shape:
        raise ValueError("out must have the query's shape")
    need = kv_int4_attention_workspace_bytes(Hq, H, d, S, max_seq_len, segment_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(_one_device(query, kv_cache, block_tables, seq_lens, query_start_loc, out, workspace)):
        st = load().kv_int8_paged_attention(query.data_ptr(), _DTYPES[query.dtype], Nq, Hq, kv_cache.data_ptr(), NB,
                                          H, d, bs, block_tables.data_ptr(), block_tables.shape[1],
                                          seq_lens.data_ptr(), query_start_loc.data_ptr(), S, max_query_len,
                                          max_seq_len, float(softmax_scale), segment_len, out.data_ptr(),
                                          _DTYPES[out.dtype], ws_ptr, ws_bytes, _stream(stream))
    _check("kv_int8_paged_attention", st)
    return out


def kv_int2_paged_attention(query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                            seq_lens: torch.Tensor, query_start_loc: torch.Tensor, softmax_scale: float,
                            rht_signs: torch.Tensor, max_query_len: int, max_seq_len: int, out=None,
                            out_dtype=None, segment_len: int = 0, workspace=None, stream=None) -> torch.Tensor:
    """Decode attention of ``query`` [Nq, Hq, d] (one query token per sequence) over the INT2
    Lloyd-Max cache; returns ``out``.  The workspace size is the INT4 call's."""
    _cuda(query, "query", (torch.float16, torch.bfloat16))
    _cuda(kv_cache, "kv_cache", (torch.uint8,))
    _cuda(block_tables, "block_tables", (torch.int32,))
    _cuda(seq_lens, "seq_lens", (torch.int32,))
    _cuda(query_start_loc, "query_start_loc", (torch.int32,))
    _cuda(rht_signs, "rht_signs", (torch.float32,))
    Nq, Hq, d = query.shape
    NB, two, bs, H, rb = kv_cache.shape
    S = seq_lens.shape[0]
    if two != 2 or rb != kv_int2_row_bytes(d) or rht_signs.shape != (d,):
        raise ValueError("kv_cache / rht_signs do not match the query's head size")
    if query_start_loc.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks] and query_start_loc [num_seqs + 1]")
    if out is None:
        out = torch.empty((Nq, Hq, d), dtype=out_dtype or query.dtype, device=query.device)
    _cuda(out, "out", tuple(_DTYPES))
    if out.shape != query.shape:
        raise ValueError("out must have the query's shape")
    need = kv_int4_attention_workspace_bytes(Hq, H, d, S, max_seq_len, segment_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(_one_device(query, kv_cache, block_tables, seq_lens, query_start_loc, rht_signs, out,
                                       workspace)):
        st = load().kv_int2_paged_attention(query.data_ptr(), _DTYPES[query.dtype], Nq, Hq, kv_cache.data_ptr(), NB,
                                          H, d, bs, block_tables.data_ptr(), block_tables.shape[1],
                                          seq_lens.data_ptr(), query_start_loc.data_ptr(), S, max_query_len,
                                          max_seq_len, float(softmax_scale), rht_signs.data_ptr(), segment_len,
                                          out.data_ptr(), _DTYPES[out.dtype], ws_ptr, ws_bytes, _stream(stream))
    _check("kv_int2_paged_attention", st)
    return out


def kv_int4_read_device_status(stream=None) -> dict:
    """Synchronise the stream and return the device's status counters by name."""
    buf = (ctypes.c_uint32 * _STAT_COUNT)()
    _check("kv_int4_read_device_status", load().kv_int4_read_device_status(buf, _stream(stream)))
    return {name: int(buf[i]) for i, name in enumerate(STAT_NAMES)}


def kv_int4_clear_device_status(stream=None) -> None:
    _check("kv_int4_clear_device_status", load().kv_int4_clear_device_status(_stream(stream)))


def kv_int4_selftest_wait_timeout(timeout_ns: int = 5_000_000, stream=None) -> None:
    """Run the bounded-wait diagnostic (a wait nothing completes); it records one wait_timeout."""
    _check("kv_int4_selftest_wait_timeout", load().kv_int4_selftest_wait_timeout(int(timeout_ns), _stream(stream)))
