"""Python loader for the fp64 CPU oracle (oracle/deft_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use this module; the library's product path
never does.  The oracle shares no code with the CUDA library.

build() compiles deft_oracle.c with gcc (OpenMP when available) into
oracle/_build/libdeft_oracle.so; load() builds on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "deft_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libdeft_oracle.so")

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source `src` into the shared library `out`."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """The default oracle library (built on first use), or the one at `path`."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_paths.argtypes = [P, i32, P, i32, P, P, i64]
    lib.oracle_paths.restype = i64
    lib.oracle_cover.argtypes = [P, i32, P, i32, P]
    lib.oracle_cover.restype = ctypes.c_int
    lib.oracle_token_counts.argtypes = [P, P, i32, P, P, i32, P, P]
    lib.oracle_token_counts.restype = ctypes.c_int
    lib.oracle_tree_attn_f64.argtypes = [P, P, P, P, P, i32, P, P, i32, P, P, i32, P, i32,
                                         i32, i32, i32, f64, P, P, i32]
    lib.oracle_tree_attn_f64.restype = ctypes.c_int
    lib.oracle_tree_attn_pieces_f64.argtypes = [P, P, P, P, P, i32, P, P, i32, P, P, i32,
                                                i32, i32, i32, f64, P, i64, P, P]
    lib.oracle_tree_attn_pieces_f64.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def paths(parent, query_node, num_nodes: Optional[int] = None, lib=None):
    """List of root-to-node paths (inclusive), one per query."""
    lib = lib or load()
    parent, query_node = _i32(parent), _i32(query_node)
    n = int(parent.shape[0]) if num_nodes is None else num_nodes
    nq = int(query_node.shape[0])
    off = np.zeros(nq + 1, dtype=np.int64)
    cap = max(1, n * max(nq, 1))
    nodes = np.zeros(cap, dtype=np.int32)
    total = lib.oracle_paths(_p(parent), n, _p(query_node), nq, _p(off), _p(nodes), cap)
    if total < 0:
        raise ValueError(f"oracle_paths failed ({total})")
    return [nodes[off[q]:off[q + 1]].tolist() for q in range(nq)]


def cover(parent, query_node, lib=None) -> np.ndarray:
    """uint64 [N, ceil(Q/64)] coverage bitsets."""
    lib = lib or load()
    parent, query_node = _i32(parent), _i32(query_node)
    n, nq = int(parent.shape[0]), int(query_node.shape[0])
    words = (nq + 63) // 64
    out = np.zeros((n, max(words, 1)), dtype=np.uint64)
    if lib.oracle_cover(_p(parent), n, _p(query_node), nq, _p(out)) != 0:
        raise ValueError("oracle_cover failed")
    return out[:, :words]


def _pos(query_pos):
    return None if query_pos is None else _i32(query_pos)


def token_counts(parent, node_len, query_node, query_pos=None, lib=None):
    """(unique tokens on any path, sum over queries of path tokens); a query
    with query_pos[q] >= 0 attends tokens 0..query_pos[q] of its own node."""
    lib = lib or load()
    parent, node_len, query_node = _i32(parent), _i32(node_len), _i32(query_node)
    pos = _pos(query_pos)
    u = np.zeros(1, dtype=np.int64)
    v = np.zeros(1, dtype=np.int64)
    rc = lib.oracle_token_counts(_p(parent), _p(node_len), int(parent.shape[0]), _p(query_node),
                                 _p(pos), int(query_node.shape[0]), _p(u), _p(v))
    if rc != 0:
        raise ValueError("oracle_token_counts failed")
    return int(u[0]), int(v[0])


def tree_attn(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, node_page_off,
              page_id, page_size: int, parent, node_len, query_node, num_q_heads: int,
              num_kv_heads: int, head_dim: int, scale: float,
              query_subset: Optional[Sequence[int]] = None, threads: int = 0, lib=None,
              query_pos=None):
    """fp64 tree attention.  q_bits/k_bits/v_bits are uint16 bf16 bit arrays
    in the library's layouts.  Returns (out [n, Hq, d], lse [n, Hq]) where n
    is the number of queries (or of `query_subset`).  query_pos: per query,
    the token of its node it sits at (-1 or None: the node's last)."""
    lib = lib or load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    node_page_off, page_id = _i32(node_page_off), _i32(page_id)
    parent, node_len, query_node = _i32(parent), _i32(node_len), _i32(query_node)
    nq = int(query_node.shape[0])
    sub = None if query_subset is None else _i32(query_subset)
    nsel = nq if sub is None else int(sub.shape[0])
    out = np.zeros((nsel, num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros((nsel, num_q_heads), dtype=np.float64)
    pos = _pos(query_pos)
    rc = lib.oracle_tree_attn_f64(_p(q_bits), _p(k_bits), _p(v_bits), _p(node_page_off),
                                  _p(page_id), page_size, _p(parent), _p(node_len),
                                  int(parent.shape[0]), _p(query_node), _p(pos), nq, _p(sub), nsel,
                                  num_q_heads, num_kv_heads, head_dim, float(scale), _p(out),
                                  _p(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_tree_attn_f64 failed")
    return out, lse


def tree_attn_pieces(q_bits, k_bits, v_bits, node_page_off, page_id, page_size: int, parent,
                     node_len, query_node, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     scale: float, cut: np.ndarray, lib=None, query_pos=None):
    """The split-and-merge form: every query's token sequence is cut before
    each position i with cut[i] != 0, pieces are merged by lse weight."""
    lib = lib or load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    node_page_off, page_id = _i32(node_page_off), _i32(page_id)
    parent, node_len, query_node = _i32(parent), _i32(node_len), _i32(query_node)
    cut = np.ascontiguousarray(cut, dtype=np.uint8)
    nq = int(query_node.shape[0])
    out = np.zeros((nq, num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros((nq, num_q_heads), dtype=np.float64)
    pos = _pos(query_pos)
    rc = lib.oracle_tree_attn_pieces_f64(_p(q_bits), _p(k_bits), _p(v_bits), _p(node_page_off),
                                         _p(page_id), page_size, _p(parent), _p(node_len),
                                         int(parent.shape[0]), _p(query_node), _p(pos), nq, num_q_heads,
                                         num_kv_heads, head_dim, float(scale), _p(cut),
                                         int(cut.shape[0]), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_tree_attn_pieces_f64 failed")
    return out, lse


def max_threads() -> int:
    return int(load().oracle_max_threads())
