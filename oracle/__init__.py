"""fp64 CPU oracle for paged-attention decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product library
(``paged_kv_decode_v2_gb300``) never imports it, and it never imports the
product library: the two share no code.  The only thing both sides use is the
seeded input generator in ``workloads``.

Contents
  * ``pa_oracle.c`` (built into ``libpa_oracle.so`` by :func:`build`):
    the definition of the decode output, the pages' phase-1 partition
    statistics and the pages' phase-2 log-sum-exp merge, all in double.
  * :mod:`oracle.brute`: a pure-Python, loop-by-loop restatement of the same
    definition for tiny inputs, used to cross-check the C code.

Sources (web pages of the project_6 fork): the "paged_attention_v2_pytorch.py"
commit list (commit 9cb7f9d, "Implementation": Phase 1 and Phase 2; commit
15ef28e, "Key changes": batched block gather and GQA broadcast) and the
"paged_attn.py" commit 490ff98 (the {m, l, o} accumulator paragraph).

Inputs are raw 16-bit storage patterns (numpy ``uint16``) plus int32 tables;
outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")

F16 = 0
BF16 = 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``src`` (default pa_oracle.c) into a shared library (portable C11, no -march)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw 16-bit patterns (uint16 or float16), got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class Problem:
    """One decode problem in the paged layout (numpy views, no copies of the caches).

    query is [S, H, D] (one new token per sequence) or [S, Q, H, D] (Q new
    tokens per sequence, each attending to its causal prefix).
    """

    def __init__(self, query, key_cache, value_cache, block_tables, seq_lens, scale, dtype):
        self.query = _u16(query)            # [S, H, D] or [S, Q, H, D]
        self.key_cache = _u16(key_cache)    # [num_blocks, KV, bs, D]
        self.value_cache = _u16(value_cache)
        self.block_tables = _i32(block_tables)  # [S, max_blocks]
        self.seq_lens = _i32(seq_lens)          # [S]
        self.scale = float(scale)
        self.dtype = int(dtype)
        if self.query.ndim == 4:
            S, Q, H, D = self.query.shape
        else:
            (S, H, D), Q = self.query.shape, 1
        self.Q = Q
        nb, KV, bs, D2 = self.key_cache.shape
        if D2 != D or self.value_cache.shape != self.key_cache.shape:
            raise ValueError("cache / query shape mismatch")
        if self.block_tables.ndim != 2 or self.block_tables.shape[0] != S:
            raise ValueError("block_tables must be [num_seqs, max_blocks]")
        self.S, self.H, self.D, self.num_blocks, self.KV, self.bs = S, H, D, nb, KV, bs
        self.max_blocks = self.block_tables.shape[1]

    @classmethod
    def from_arrays(cls, arrays: dict) -> "Problem":
        return cls(arrays["query"], arrays["key_cache"], arrays["value_cache"],
                   arrays["block_tables"], arrays["seq_lens"], arrays["scale"], arrays["dtype"])

    def _args(self):
        return [_ptr(self.query), _ptr(self.key_cache), _ptr(self.value_cache),
                _ptr(self.block_tables), _ptr(self.seq_lens), self.S, self.Q, self.H, self.KV,
                self.D, self.num_blocks, self.bs, self.max_blocks, self.scale, self.dtype]

    def out_shape(self):
        return (self.S, self.Q, self.H, self.D) if self.query.ndim == 4 else (self.S, self.H, self.D)


def _pairs(problem: Problem, pairs):
    """pairs are (row, head) with row = b * Q + i (row = b when Q = 1)."""
    if pairs is None:
        return None, problem.S * problem.Q * problem.H
    arr = _i32(pairs).reshape(-1, 2)
    return arr, arr.shape[0]


class OracleLib:
    """ctypes view of one build of pa_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.pa_oracle_decode_mq.restype = I
        lib.pa_oracle_decode_mq.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, P, I, P, I]
        lib.pa_oracle_partition_stats_mq.restype = I
        lib.pa_oracle_partition_stats_mq.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D, I,
                                                     I, P, I, I, P, P, P, P, I]
        lib.pa_oracle_merge.restype = I
        lib.pa_oracle_merge.argtypes = [P, P, P, I, I, P]
        lib.pa_oracle_decode_scalar.restype = D
        lib.pa_oracle_decode_scalar.argtypes = [ctypes.c_uint16, I]
        self.lib = lib
        self.path = path

    def decode(self, problem: Problem, pairs=None, num_threads: int = 0) -> np.ndarray:
        """Unpartitioned softmax decode.  Returns the query's shape (pairs=None) or [n, D] doubles."""
        arr, n = _pairs(problem, pairs)
        out = np.empty((n, problem.D), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_mq(*problem._args(), None if arr is None else _ptr(arr), n,
                                          _ptr(out), int(num_threads))
        if rc:
            raise RuntimeError(f"pa_oracle_decode failed with code {rc}")
        return out.reshape(problem.out_shape()) if arr is None else out

    def partition_stats(self, problem: Problem, partition_size: int, pairs=None,
                        max_partitions=None, num_threads: int = 0):
        """Phase 1: (o_p [n, NP, D], m_p [n, NP], l_p [n, NP], num_p [n]); unused slots are NaN."""
        arr, n = _pairs(problem, pairs)
        if max_partitions is None:
            max_partitions = max(1, -(-problem.max_blocks * problem.bs // partition_size))
        o = np.full((n, max_partitions, problem.D), np.nan)
        m = np.full((n, max_partitions), np.nan)
        l = np.full((n, max_partitions), np.nan)
        num = np.zeros(n, dtype=np.int32)
        rc = self.lib.pa_oracle_partition_stats_mq(*problem._args(), int(partition_size),
                                                None if arr is None else _ptr(arr), n,
                                                int(max_partitions), _ptr(o), _ptr(m), _ptr(l),
                                                _ptr(num), int(num_threads))
        if rc:
            raise RuntimeError(f"pa_oracle_partition_stats failed with code {rc}")
        return o, m, l, num

    def merge(self, o_p, m_p, l_p) -> np.ndarray:
        """Phase 2 for one (seq, head): o_p [np, D], m_p [np], l_p [np] -> out [D]."""
        o_p = np.ascontiguousarray(o_p, dtype=np.float64)
        m_p = np.ascontiguousarray(m_p, dtype=np.float64)
        l_p = np.ascontiguousarray(l_p, dtype=np.float64)
        n = m_p.shape[0]
        D = o_p.shape[-1]
        out = np.empty(D, dtype=np.float64)
        rc = self.lib.pa_oracle_merge(_ptr(o_p), _ptr(m_p), _ptr(l_p), n, D, _ptr(out))
        if rc:
            raise RuntimeError(f"pa_oracle_merge failed with code {rc}")
        return out

    def decode_scalar(self, bits: int, dtype: int) -> float:
        """The oracle's exact decoding of one 16-bit storage pattern."""
        return float(self.lib.pa_oracle_decode_scalar(int(bits) & 0xFFFF, int(dtype)))


_default = None


def lib() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def decode(problem: Problem, pairs=None, num_threads: int = 0) -> np.ndarray:
    return lib().decode(problem, pairs, num_threads)


def partition_stats(problem: Problem, partition_size: int, pairs=None, max_partitions=None,
                    num_threads: int = 0):
    return lib().partition_stats(problem, partition_size, pairs, max_partitions, num_threads)


def merge(o_p, m_p, l_p) -> np.ndarray:
    return lib().merge(o_p, m_p, l_p)


def decode_scalar(bits: int, dtype: int) -> float:
    return lib().decode_scalar(bits, dtype)
