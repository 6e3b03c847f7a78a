"""ctypes binding of libpa_decode.so (the C ABI in include/pa_decode.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory
and streams); their data pointers and the current CUDA stream are passed
through.  If the shared library is missing the import fails loudly -- there
is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_decode.so")

PA_F16 = 0
PA_BF16 = 1
PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4
PA_STATUS_BAD_BLOCK_ID = 1
PA_STATUS_BAD_SEQ_LEN = 2
PA_STATUS_TIMEOUT = 4

_DTYPE = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({status_string(code)})")
        self.code = code


def load() -> ctypes.CDLL:
    """Load the in-tree library (built by ``paged_kv_decode_v2_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: run paged_kv_decode_v2_gb300.build.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    attn = [P, P, P, P, P, I, I, I, I, I, I, I, I, F]
    lib.pa_v2_num_partitions.argtypes = [I, I]
    lib.pa_v2_num_partitions.restype = I
    lib.pa_v2_workspace_bytes.argtypes = [I, I, I, I]
    lib.pa_v2_workspace_bytes.restype = S
    lib.pa_decode_v2.argtypes = attn + [I, I, P, P, P, P, I, P, P]
    lib.pa_decode_v2.restype = I
    lib.pa_decode_v2_fused.argtypes = attn + [I, I, P, P, P, P, I, P, P, P]
    lib.pa_decode_v2_fused.restype = I
    lib.pa_decode_v2_phase1.argtypes = attn + [I, I, P, P, P, I, P, P]
    lib.pa_decode_v2_phase1.restype = I
    lib.pa_decode_v2_phase2.argtypes = [P, I, I, I, I, I, I, P, P, P, I, P, P, P]
    lib.pa_decode_v2_phase2.restype = I
    lib.pa_decode_v1.argtypes = attn + [I, P, P, P]
    lib.pa_decode_v1.restype = I
    attn_mq = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F]
    lib.pa_decode_v2_mq.argtypes = attn_mq + [I, I, P, P, P, P, I, P, P]
    lib.pa_decode_v2_mq.restype = I
    lib.pa_decode_v1_mq.argtypes = attn_mq + [I, P, P, P]
    lib.pa_decode_v1_mq.restype = I
    lib.pa_decode.argtypes = attn + [I, I, P, P, P, P, I, P, P]
    lib.pa_decode.restype = I
    lib.pa_decode_choose.argtypes = [I, I, I, I]
    lib.pa_decode_choose.restype = I
    lib.pa_decode_mq.argtypes = attn_mq + [I, I, P, P, P, P, I, P, P]
    lib.pa_decode_mq.restype = I
    lib.pa_decode_mq_choose.argtypes = [I, I, I, I, I, I, I]
    lib.pa_decode_mq_choose.restype = I
    lib.pa_decode_mq_partition.argtypes = [I, I, I, I, I, I, I]
    lib.pa_decode_mq_partition.restype = I
    lib.pa_status_string.argtypes = [I]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_set_launch_config.argtypes = [I, I]
    lib.pa_set_launch_config.restype = I
    lib.pa_set_rows_kernel.argtypes = [I]
    lib.pa_set_rows_kernel.restype = I
    lib.pa_set_merge_form.argtypes = [I]
    lib.pa_set_merge_form.restype = I
    lib.pa_selftest_wait_timeout.argtypes = [P, ctypes.c_longlong, P]
    lib.pa_selftest_wait_timeout.restype = I
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().pa_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, rc: int):
    if rc != PA_OK:
        raise PagedAttentionError(fn, rc)


def _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale):
    if query.dtype not in _DTYPE or key_cache.dtype != query.dtype or value_cache.dtype != query.dtype:
        raise TypeError("query / key_cache / value_cache must share one dtype: float16 or bfloat16")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    for t in (query, key_cache, value_cache, block_tables, seq_lens):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    S, H, D = query.shape
    nb, KV, bs, D2 = key_cache.shape
    if D2 != D or tuple(value_cache.shape) != tuple(key_cache.shape):
        raise ValueError("cache shapes must be [num_blocks, num_kv_heads, block_size, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape != (S,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
    return [_ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), _ptr(seq_lens),
            S, H, KV, D, nb, bs, block_tables.shape[1], int(max_seq_len_hint), float(scale)]


def _shape_args_mq(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale):
    """Arguments of the _mq entry points: query [S, Q, H, D]."""
    if query.dim() != 4:
        raise ValueError("query must be [num_seqs, q_len, num_heads, head_dim]")
    S, Q, H, D = query.shape
    a = _shape_args(query.view(S, Q * H, D), key_cache, value_cache, block_tables, seq_lens,
                    max_seq_len_hint, scale)
    return a[:5] + [S, Q, H] + a[7:]


def num_partitions(max_seq_len: int, partition_size: int) -> int:
    return load().pa_v2_num_partitions(int(max_seq_len), int(partition_size))


def workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_num_partitions: int) -> int:
    return load().pa_v2_workspace_bytes(num_seqs, num_heads, head_dim, max_num_partitions)


def alloc_workspace(num_seqs: int, num_heads: int, head_dim: int, max_num_partitions: int,
                    device="cuda", q_len: int = 1):
    """Allocate (tmp_output, exp_sums, max_logits) once, to be reused across calls.

    Shapes [S, H, NP, D] / [S, H, NP], or [S, Q, H, NP, D] / [S, Q, H, NP] for q_len Q > 1.
    """
    lead = (num_seqs, num_heads) if q_len == 1 else (num_seqs, q_len, num_heads)
    tmp = torch.empty(lead + (max_num_partitions, head_dim), dtype=torch.float32, device=device)
    es = torch.empty(lead + (max_num_partitions,), dtype=torch.float32, device=device)
    ml = torch.empty_like(es)
    return tmp, es, ml


def pa_decode_v2(query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
                 out, tmp_output, exp_sums, max_logits, max_seq_len_hint=0, status=None,
                 stream=None):
    lib = load()
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    rc = lib.pa_decode_v2(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out),
                          _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits),
                          tmp_output.shape[2], _ptr(status), _stream(stream))
    _check("pa_decode_v2", rc)
    return out


def alloc_counters(num_seqs: int, num_kv_heads: int, device="cuda"):
    """The zeroed ticket counters pa_decode_v2_fused needs: [num_seqs, num_kv_heads] int32.
    Every completed call leaves them zero again, so they are allocated once."""
    return torch.zeros((num_seqs, num_kv_heads), dtype=torch.int32, device=device)


def pa_decode_v2_fused(query, key_cache, value_cache, block_tables, seq_lens, scale,
                       partition_size, out, tmp_output, exp_sums, max_logits, counters,
                       max_seq_len_hint=0, status=None, stream=None):
    """pa_decode_v2 in one kernel: the last CTA of each (sequence, KV head) merges."""
    lib = load()
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    if counters.dtype != torch.int32 or not counters.is_cuda or counters.numel() < args[5] * args[7]:
        raise ValueError("counters must be a CUDA int32 tensor of num_seqs * num_kv_heads zeros")
    rc = lib.pa_decode_v2_fused(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out),
                                _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits),
                                tmp_output.shape[2], _ptr(counters), _ptr(status), _stream(stream))
    _check("pa_decode_v2_fused", rc)
    return out


def pa_decode_v2_phase1(query, key_cache, value_cache, block_tables, seq_lens, scale,
                        partition_size, tmp_output, exp_sums, max_logits, max_seq_len_hint=0,
                        status=None, stream=None):
    lib = load()
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    rc = lib.pa_decode_v2_phase1(*args, int(partition_size), _DTYPE[query.dtype],
                                 _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits),
                                 tmp_output.shape[2], _ptr(status), _stream(stream))
    _check("pa_decode_v2_phase1", rc)


def pa_decode_v2_phase2(seq_lens, max_seq_len, partition_size, tmp_output, exp_sums, max_logits,
                        out, status=None, stream=None):
    lib = load()
    S, H, NP, D = tmp_output.shape
    rc = lib.pa_decode_v2_phase2(_ptr(seq_lens), S, H, D, int(max_seq_len), int(partition_size),
                                 _DTYPE[out.dtype], _ptr(tmp_output), _ptr(exp_sums),
                                 _ptr(max_logits), NP, _ptr(out), _ptr(status), _stream(stream))
    _check("pa_decode_v2_phase2", rc)
    return out


def pa_decode_v2_mq(query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
                    out, tmp_output, exp_sums, max_logits, max_seq_len_hint=0, status=None,
                    stream=None):
    """Several new tokens per sequence: query / out [S, Q, H, D], intermediates [S, Q, H, NP, ...]."""
    lib = load()
    args = _shape_args_mq(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint,
                          scale)
    rc = lib.pa_decode_v2_mq(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out),
                             _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits),
                             tmp_output.shape[-2], _ptr(status), _stream(stream))
    _check("pa_decode_v2_mq", rc)
    return out


def pa_decode_v1_mq(query, key_cache, value_cache, block_tables, seq_lens, scale, out,
                    max_seq_len_hint=0, status=None, stream=None):
    lib = load()
    args = _shape_args_mq(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint,
                          scale)
    rc = lib.pa_decode_v1_mq(*args, _DTYPE[query.dtype], _ptr(out), _ptr(status), _stream(stream))
    _check("pa_decode_v1_mq", rc)
    return out


def pa_decode_mq(query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
                 out, tmp_output, exp_sums, max_logits, max_seq_len_hint=0, status=None,
                 stream=None):
    """Several new tokens per sequence, V1 or V2 as pa_decode_mq_choose picks."""
    lib = load()
    args = _shape_args_mq(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint,
                          scale)
    rc = lib.pa_decode_mq(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out),
                          _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits),
                          tmp_output.shape[-2], _ptr(status), _stream(stream))
    _check("pa_decode_mq", rc)
    return out


def pa_decode_mq_choose(num_seqs: int, q_len: int, num_heads: int, num_kv_heads: int,
                        head_dim: int, max_seq_len: int, partition_size: int) -> int:
    r = load().pa_decode_mq_choose(num_seqs, q_len, num_heads, num_kv_heads, head_dim,
                                   max_seq_len, partition_size)
    if r < 0:
        raise PagedAttentionError("pa_decode_mq_choose", -r)
    return r


def pa_decode_mq_partition(num_seqs: int, q_len: int, num_heads: int, num_kv_heads: int,
                           head_dim: int, max_seq_len: int, partition_size: int) -> int:
    """Partition size pa_decode_mq runs V2 with (0 when it runs V1)."""
    r = load().pa_decode_mq_partition(num_seqs, q_len, num_heads, num_kv_heads, head_dim,
                                      max_seq_len, partition_size)
    if r < 0:
        raise PagedAttentionError("pa_decode_mq_partition", -r)
    return r


def pa_decode_v1(query, key_cache, value_cache, block_tables, seq_lens, scale, out,
                 max_seq_len_hint=0, status=None, stream=None):
    lib = load()
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    rc = lib.pa_decode_v1(*args, _DTYPE[query.dtype], _ptr(out), _ptr(status), _stream(stream))
    _check("pa_decode_v1", rc)
    return out


def pa_decode(query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size, out,
              tmp_output, exp_sums, max_logits, max_seq_len_hint=0, status=None, stream=None):
    lib = load()
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    rc = lib.pa_decode(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out),
                       _ptr(tmp_output), _ptr(exp_sums), _ptr(max_logits), tmp_output.shape[2],
                       _ptr(status), _stream(stream))
    _check("pa_decode", rc)
    return out


def pa_decode_choose(num_seqs: int, num_kv_heads: int, max_seq_len: int, partition_size: int) -> int:
    r = load().pa_decode_choose(num_seqs, num_kv_heads, max_seq_len, partition_size)
    if r < 0:
        raise PagedAttentionError("pa_decode_choose", -r)
    return r


def pa_set_launch_config(warps_per_cta: int = 0, stages_per_warp: int = 0) -> None:
    _check("pa_set_launch_config", load().pa_set_launch_config(warps_per_cta, stages_per_warp))


def pa_set_rows_kernel(mode: int = 0) -> None:
    """0: by query rows per KV head; 1: always mma.sync; 2: always tcgen05; 3: tcgen05, one
    query tile per CTA; 4: tcgen05, two query tiles per CTA; 5: the CUDA-core (SIMT) kernel
    up to 8 rows per KV head, else as 0; 6: tcgen05, one query tile per CTA with the whole
    128-row Q tile stored (modes 0 and 3 store 64 rows for KV heads of at most 64 rows)."""
    _check("pa_set_rows_kernel", load().pa_set_rows_kernel(mode))


def pa_set_merge_form(form: int = 0) -> None:
    """Phase 2's form: 0 by rule; 1 a CTA per (head, row, slice of head_dim); 2 a warp per
    (row, head)."""
    _check("pa_set_merge_form", load().pa_set_merge_form(form))


def pa_selftest_wait_timeout(status, limit_ns: int, stream=None) -> None:
    _check("pa_selftest_wait_timeout",
           load().pa_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)))


def pa_decode_v2_static(query, key_cache, value_cache, block_tables, seq_lens, scale,
                        partition_size, out, max_seq_len_hint=0, status=None, stream=None):
    """pa_decode_v2 with the intermediates kept in the library's own device array.

    For callers that cannot allocate device memory themselves; see
    pa_decode_v2_static in include/pa_decode.h for the size limit and for why
    concurrent calls must not overlap on the GPU.
    """
    lib = load()
    fn = lib.pa_decode_v2_static
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, P, P]
    fn.restype = I
    args = _shape_args(query, key_cache, value_cache, block_tables, seq_lens, max_seq_len_hint, scale)
    rc = fn(*args, int(partition_size), _DTYPE[query.dtype], _ptr(out), _ptr(status),
            _stream(stream))
    _check("pa_decode_v2_static", rc)
    return out
