"""CPU oracle for the batched speculative-decoding verifier (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  The GPU library never imports, links or calls it, and the two share
no code: the arithmetic lives in ``sv_oracle.c`` (plain C, fp64), written from the pages'
definitions and cited there function by function.  This module only builds that file with
gcc and marshals numpy arrays into it.

Dtype codes: 0 = bf16 (passed as uint16 bit patterns), 1 = fp32, 2 = fp64.
Status codes per request: 0 ok, 1 draft/node token outside [-1, V), 2 a row holding NaN,
+inf or no finite logit, 3 malformed tree, 4 duplicate sibling tokens (target-only trees).
When a request has several faults the largest code is reported.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsvoracle.so")
_lib = None
_lock = threading.Lock()

DT_BF16, DT_FP32, DT_FP64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile sv_oracle.c into libsvoracle.so beside it (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I32P, F64P = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
        i32, i64, u64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.svo_philox4x32_10.argtypes = [P, P, P]
        lib.svo_philox4x32_10.restype = None
        lib.svo_u01.argtypes = [ctypes.c_uint32]
        lib.svo_u01.restype = f64
        lib.svo_uniform_pair.argtypes = [u64, u64, ctypes.c_uint32, ctypes.c_uint32, F64P, F64P]
        lib.svo_uniform_pair.restype = None
        lib.svo_softmax_row.argtypes = [P, i32, i64, i64, f64, P]
        lib.svo_softmax_row.restype = i32
        lib.svo_argmax_row.argtypes = [P, i32, i64, i64, I32P]
        lib.svo_argmax_row.restype = i32
        lib.svo_chain_core.argtypes = [P, P, P, i32, i64, P, P, P, I32P, I32P, P, P]
        lib.svo_chain_core.restype = i32
        lib.svo_tree_check.argtypes = [P, P, i32, i64, i32]
        lib.svo_tree_check.restype = i32
        lib.svo_tree_core.argtypes = [P, P, P, P, i32, i64, i32, P, P, P, P, I32P, I32P, P]
        lib.svo_tree_core.restype = i32
        lib.svo_verify_greedy.argtypes = [P, i32, P, i32, i32, i64, P, i32, P, P, P]
        lib.svo_verify_greedy.restype = i32
        lib.svo_verify_rejection.argtypes = [P, i32, P, P, i32, i32, i64, f64, u64, u64, P, i32,
                                             P, P, P, P, P]
        lib.svo_verify_rejection.restype = i32
        lib.svo_verify_tree.argtypes = [P, i32, P, P, i32, i32, i64, i32, f64, u64, u64, P, i32,
                                        P, P, P, P, P]
        lib.svo_verify_tree.restype = i32
        lib.svo_block_core.argtypes = [P, P, P, i32, i64, P, P, P, I32P, I32P, P]
        lib.svo_block_core.restype = i32
        lib.svo_verify_block.argtypes = [P, i32, P, P, i32, i32, i64, f64, u64, u64, P, i32,
                                         P, P, P, P]
        lib.svo_verify_block.restype = i32
        lib.svo_grid_chain_first_token.argtypes = [P, P, P, i64, i32, P, F64P]
        lib.svo_grid_chain_first_token.restype = i32
        lib.svo_grid_tree_first_token.argtypes = [P, P, i32, i64, i32, P, F64P]
        lib.svo_grid_tree_first_token.restype = i32
        lib.svo_grid_tree_first_token_t.argtypes = [P, P, i32, i64, i32, f64, f64, P, F64P]
        lib.svo_grid_tree_first_token_t.restype = i32
        lib.svo_chain_core_t.argtypes = [P, P, P, i32, i64, P, P, f64, f64, P, I32P, I32P, P, P]
        lib.svo_chain_core_t.restype = i32
        lib.svo_verify_ex.argtypes = [P, i32, P, P, i32, i32, i64, P, f64, f64, P, P, u64, u64, P,
                                      i32, P, P, P, P, P]
        lib.svo_verify_ex.restype = i32
        lib.svo_verify_tree_ex.argtypes = [P, i32, P, P, i32, i32, i64, P, f64, f64, P, P, u64, u64,
                                           P, i32, P, P, P, P, P]
        lib.svo_filter_row.argtypes = [P, i32, i64, i64, i32, f64, P, I32P]
        lib.svo_filter_row.restype = i32
        lib.svo_verify_tree_ex.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits(logits):
    """Accept a numpy array (uint16 = bf16 bits, float32, float64) and return (array, code)."""
    a = np.ascontiguousarray(logits)
    if a.dtype == np.uint16:
        return a, DT_BF16
    if a.dtype == np.float32:
        return a, DT_FP32
    if a.dtype == np.float64:
        return a, DT_FP64
    raise TypeError(f"unsupported logits dtype {a.dtype}")


def _req_ids(req_ids, B):
    if req_ids is None:
        return np.arange(B, dtype=np.int32)
    return _c(req_ids, np.int32)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")


# ---------------------------------------------------------------------------------------
# RNG
# ---------------------------------------------------------------------------------------
def philox4x32_10(ctr, key):
    """Philox4x32-10 of one 4-word counter and 2-word key -> 4 uint32 words."""
    lib = _load()
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.svo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def u01(x: int) -> float:
    return _load().svo_u01(int(x))


def uniform_pair(seed: int, offset: int, slot: int, request: int):
    lib = _load()
    u, v = ctypes.c_double(), ctypes.c_double()
    lib.svo_uniform_pair(seed, offset, slot, request, ctypes.byref(u), ctypes.byref(v))
    return u.value, v.value


# ---------------------------------------------------------------------------------------
# Rows
# ---------------------------------------------------------------------------------------
def softmax_rows(logits, T: float):
    """p = softmax(l / T) for every row of a [rows, V] array (fp64 out); raises on bad rows."""
    lib = _load()
    a, dt = _logits(logits)
    a2 = a.reshape(-1, a.shape[-1])
    rows, V = a2.shape
    p = np.zeros((rows, V), np.float64)
    for r in range(rows):
        st = lib.svo_softmax_row(_ptr(a2), dt, r, V, float(T), _ptr(p[r]))
        if st != 0:
            raise ValueError(f"row {r} invalid (status {st})")
    return p.reshape(a.shape)


def argmax_rows(logits):
    lib = _load()
    a, dt = _logits(logits)
    a2 = a.reshape(-1, a.shape[-1])
    rows, V = a2.shape
    out = np.zeros(rows, np.int32)
    for r in range(rows):
        idx = ctypes.c_int32()
        st = lib.svo_argmax_row(_ptr(a2), dt, r, V, ctypes.byref(idx))
        if st != 0:
            raise ValueError(f"row {r} invalid (status {st})")
        out[r] = idx.value
    return out.reshape(a.shape[:-1])


# ---------------------------------------------------------------------------------------
# Cores with explicit uniforms (used by the self-tests)
# ---------------------------------------------------------------------------------------
def chain_core(p, q, drafts, u, v, thr_single=1.0, thr_acc=1.0):
    """One request: p [(k+1), V] fp64, q [k, V] fp64 or None, drafts [k], u/v [k+1]; thresholds
    below 1 relax the target-only test (q None)."""
    lib = _load()
    p = _c(p, np.float64)
    k1, V = p.shape
    k = k1 - 1
    q = None if q is None else _c(q, np.float64)
    d = _c(drafts, np.int32)
    u = _c(u, np.float64)
    v = _c(v, np.float64)
    tokens = np.zeros(k + 1, np.int32)
    probs = np.zeros((k + 1, 3), np.float64)
    work = np.zeros(V, np.float64)
    alen, bnd = ctypes.c_int32(), ctypes.c_int32(0)
    st = lib.svo_chain_core_t(_ptr(p), _ptr(q), _ptr(d), k, V, _ptr(u), _ptr(v), float(thr_single),
                              float(thr_acc), _ptr(tokens), ctypes.byref(alen), ctypes.byref(bnd),
                              _ptr(probs), _ptr(work))
    return dict(status=st, tokens=tokens, accept_len=alen.value, boundary=bnd.value, probs=probs)


def tree_core(p, amax, tokens, parents, mode, coin, v, V=None):
    lib = _load()
    tokens = _c(tokens, np.int32)
    parents = _c(parents, np.int32)
    N = tokens.shape[0]
    if p is not None:
        p = _c(p, np.float64)
        V = p.shape[1]
    amax = None if amax is None else _c(amax, np.int32)
    coin = None if coin is None else _c(coin, np.float64)
    v = None if v is None else _c(v, np.float64)
    ot = np.zeros(N, np.int32)
    ai = np.zeros(N, np.int32)
    work = np.zeros(V, np.float64)
    alen, bnd = ctypes.c_int32(), ctypes.c_int32(0)
    st = lib.svo_tree_core(_ptr(p), _ptr(amax), _ptr(tokens), _ptr(parents), N, V, mode,
                           _ptr(coin), _ptr(v), _ptr(ot), _ptr(ai), ctypes.byref(alen),
                           ctypes.byref(bnd), _ptr(work))
    return dict(status=st, out_tokens=ot, accept_index=ai, accept_len=alen.value,
                boundary=bnd.value)


def tree_check(tokens, parents, V, mode):
    lib = _load()
    t = _c(tokens, np.int32)
    pa = _c(parents, np.int32)
    return lib.svo_tree_check(_ptr(t), _ptr(pa), t.shape[0], V, mode)


def grid_chain_first_token(p0, q0, w, G: int):
    """Integrate one chain position over a G x G (u, v) grid, drafts weighted by w."""
    lib = _load()
    p0 = _c(p0, np.float64)
    V = p0.shape[0]
    q0 = None if q0 is None else _c(q0, np.float64)
    w = _c(w, np.float64)
    dist = np.zeros(V, np.float64)
    acc = ctypes.c_double()
    _check(lib.svo_grid_chain_first_token(_ptr(p0), _ptr(q0), _ptr(w), V, G, _ptr(dist),
                                          ctypes.byref(acc)))
    return dist, acc.value


def grid_tree_first_token(p0, child_tokens, G: int, thr_single=1.0, thr_acc=1.0):
    """Integrate one target-only tree level over a G x G (coin, v) grid; thresholds below 1
    give the relaxed rule."""
    lib = _load()
    p0 = _c(p0, np.float64)
    V = p0.shape[0]
    ct = _c(child_tokens, np.int32)
    dist = np.zeros(V, np.float64)
    acc = ctypes.c_double()
    _check(lib.svo_grid_tree_first_token_t(_ptr(p0), _ptr(ct), ct.shape[0], V, G, float(thr_single),
                                           float(thr_acc), _ptr(dist), ctypes.byref(acc)))
    return dist, acc.value


# ---------------------------------------------------------------------------------------
# Batched entry points (same semantics as the GPU library's C ABI)
# ---------------------------------------------------------------------------------------
def verify_greedy(logits, drafts, req_ids=None):
    """logits [B, k+1, V]; drafts [B, k] int32."""
    lib = _load()
    a, dt = _logits(logits)
    B, k1, V = a.shape
    k = k1 - 1
    d = _c(drafts, np.int32).reshape(B, k)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    out = np.zeros((n, k + 1), np.int32)
    alen = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_greedy(_ptr(a), dt, _ptr(d), B, k, V, _ptr(ids), n, _ptr(out),
                                 _ptr(alen), _ptr(status)))
    return dict(out_tokens=out, accept_len=alen, status=status)


def verify_rejection(logits, drafts, q, T: float, seed: int, offset: int, req_ids=None):
    """logits [B, k+1, V]; drafts [B, k]; q [B, k, V] float32 or None (one-hot drafts)."""
    lib = _load()
    a, dt = _logits(logits)
    B, k1, V = a.shape
    k = k1 - 1
    d = _c(drafts, np.int32).reshape(B, k)
    qq = None if q is None else _c(q, np.float32).reshape(B, k, V)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    out = np.zeros((n, k + 1), np.int32)
    alen = np.zeros(n, np.int32)
    probs = np.zeros((n, k + 1, 3), np.float64)
    bnd = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_rejection(_ptr(a), dt, _ptr(d), _ptr(qq), B, k, V, float(T), seed,
                                    offset, _ptr(ids), n, _ptr(out), _ptr(alen), _ptr(probs),
                                    _ptr(bnd), _ptr(status)))
    return dict(out_tokens=out, accept_len=alen, out_probs=probs, boundary=bnd, status=status)


def _opt_arrays(B, top_k, top_p):
    tk = None if top_k is None else _c(top_k, np.int32).reshape(B)
    tp = None if top_p is None else _c(top_p, np.float64).reshape(B)
    return tk, tp


def filter_row(logits, row: int, T: float, top_k: int, top_p: float):
    """Probabilities of one row of logits [rows, V] at temperature T after top-k and top-p."""
    lib = _load()
    a, dt = _logits(logits)
    V = a.shape[-1]
    p = np.zeros(V, np.float64)
    _check(lib.svo_softmax_row(_ptr(a), dt, row, V, float(T), _ptr(p)))
    bnd = ctypes.c_int32(0)
    _check(lib.svo_filter_row(_ptr(a), dt, row, V, int(top_k), float(top_p), _ptr(p), ctypes.byref(bnd)))
    return p, bnd.value


def verify_ex(logits, drafts, q, temps, seed: int, offset: int, thr_single=1.0, thr_acc=1.0,
              req_ids=None, top_k=None, top_p=None):
    """Chain verification with a temperature per request (temps [B]; 0 = greedy for that
    request), the relaxed thresholds of target-only decisions (q must be None unless both are
    1) and per-request top-k / top-p on p (top_k [B] int, 0 = off; top_p [B], 1 = off).  Same
    outputs as verify_rejection; a greedy request's out_probs are 0."""
    lib = _load()
    a, dt = _logits(logits)
    B, k1, V = a.shape
    k = k1 - 1
    d = _c(drafts, np.int32).reshape(B, k)
    qq = None if q is None else _c(q, np.float32).reshape(B, k, V)
    tt = _c(temps, np.float64).reshape(B)
    tk, tp = _opt_arrays(B, top_k, top_p)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    out = np.zeros((n, k + 1), np.int32)
    alen = np.zeros(n, np.int32)
    probs = np.zeros((n, k + 1, 3), np.float64)
    bnd = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_ex(_ptr(a), dt, _ptr(d), _ptr(qq), B, k, V, _ptr(tt), float(thr_single),
                             float(thr_acc), _ptr(tk), _ptr(tp), seed, offset, _ptr(ids), n,
                             _ptr(out), _ptr(alen), _ptr(probs), _ptr(bnd), _ptr(status)))
    return dict(out_tokens=out, accept_len=alen, out_probs=probs, boundary=bnd, status=status)


def verify_tree_ex(logits, tokens, parents, temps, seed: int, offset: int, thr_single=1.0,
                   thr_acc=1.0, req_ids=None, top_k=None, top_p=None):
    """Tree verification with a temperature per request (0 = greedy walk for that request) and
    the relaxed thresholds of the target-only walk."""
    lib = _load()
    a, dt = _logits(logits)
    B, N, V = a.shape
    t = _c(tokens, np.int32).reshape(B, N)
    pa = _c(parents, np.int32).reshape(B, N)
    tt = _c(temps, np.float64).reshape(B)
    tk, tp = _opt_arrays(B, top_k, top_p)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    ot = np.zeros((n, N), np.int32)
    ai = np.zeros((n, N), np.int32)
    alen = np.zeros(n, np.int32)
    bnd = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_tree_ex(_ptr(a), dt, _ptr(t), _ptr(pa), B, N, V, _ptr(tt),
                                  float(thr_single), float(thr_acc), _ptr(tk), _ptr(tp), seed, offset,
                                  _ptr(ids), n, _ptr(ot), _ptr(ai), _ptr(alen), _ptr(bnd), _ptr(status)))
    return dict(out_tokens=ot, accept_index=ai, accept_len=alen, boundary=bnd, status=status)


def block_core(p, q, drafts, u, v):
    """Block verification of one request from probabilities: p [k+1, V], q [k, V] or None
    (one-hot drafts), drafts [k], uniforms u, v [k+1].  Returns (tokens, accept_len, boundary)."""
    lib = _load()
    pp = _c(p, np.float64)
    k1, V = pp.shape
    k = k1 - 1
    qq = None if q is None else _c(q, np.float64).reshape(k, V)
    d = _c(drafts, np.int32).reshape(k)
    uu, vv = _c(u, np.float64), _c(v, np.float64)
    tok = np.zeros(k + 1, np.int32)
    alen = ctypes.c_int32(-1)
    bnd = ctypes.c_int32(0)
    work = np.zeros(V, np.float64)
    st = lib.svo_block_core(_ptr(pp), _ptr(qq), _ptr(d), k, V, _ptr(uu), _ptr(vv), _ptr(tok),
                            ctypes.byref(alen), ctypes.byref(bnd), _ptr(work))
    if st != 0:
        raise RuntimeError(f"oracle block core returned {st}")
    return tok, alen.value, bnd.value


def verify_block(logits, drafts, q, T: float, seed: int, offset: int, req_ids=None):
    """Block verification.  logits [B, k+1, V]; drafts [B, k]; q [B, k, V] or None (one-hot)."""
    lib = _load()
    a, dt = _logits(logits)
    B, k1, V = a.shape
    k = k1 - 1
    d = _c(drafts, np.int32).reshape(B, k)
    qq = None if q is None else _c(q, np.float32).reshape(B, k, V)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    out = np.zeros((n, k + 1), np.int32)
    alen = np.zeros(n, np.int32)
    bnd = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_block(_ptr(a), dt, _ptr(d), _ptr(qq), B, k, V, float(T), seed, offset,
                                _ptr(ids), n, _ptr(out), _ptr(alen), _ptr(bnd), _ptr(status)))
    return dict(out_tokens=out, accept_len=alen, boundary=bnd, status=status)


def verify_tree(logits, tokens, parents, mode: int, T: float, seed: int, offset: int,
                req_ids=None):
    """logits [B, N, V]; tokens, parents [B, N] int32; mode 0 greedy, 1 target-only."""
    lib = _load()
    a, dt = _logits(logits)
    B, N, V = a.shape
    t = _c(tokens, np.int32).reshape(B, N)
    pa = _c(parents, np.int32).reshape(B, N)
    ids = _req_ids(req_ids, B)
    n = ids.shape[0]
    ot = np.zeros((n, N), np.int32)
    ai = np.zeros((n, N), np.int32)
    alen = np.zeros(n, np.int32)
    bnd = np.zeros(n, np.int32)
    status = np.zeros(n, np.int32)
    _check(lib.svo_verify_tree(_ptr(a), dt, _ptr(t), _ptr(pa), B, N, V, mode, float(T), seed,
                               offset, _ptr(ids), n, _ptr(ot), _ptr(ai), _ptr(alen), _ptr(bnd),
                               _ptr(status)))
    return dict(out_tokens=ot, accept_index=ai, accept_len=alen, boundary=bnd, status=status)


# ---------------------------------------------------------------------------------------
# After tree verification: the accepted path's KV rows move to contiguous positions after the
# committed prefix, and the committed length advances by the accepted nodes plus one ("投机解码",
# section 与调度、KV 的交互, SGLang part: committed length plus the accepted count, and with
# topk > 1 the accepted path, which is not contiguous in the tree, is moved to contiguous
# positions; "Draft sources: draft models, n-gram, suffix decoding", section "SGLang's suffix
# automaton, in tree", the NGRAM decode-step walk-through: verification, then
# move_accept_tokens_to_target_kvcache).
# ---------------------------------------------------------------------------------------
KV_OK, KV_BAD_POSITION, KV_BAD_SLOT = 0, 1, 2


def kv_compact(pool, slot_table, committed, accept_index, accept_len):
    """pool [num_slots, row] or [planes, num_slots, row] (any dtype, modified in place; a plane is
    one layer's K or V); slot_table [B, max_pos] int; committed [B]; accept_index [B, N] (node 0,
    then the accepted nodes); accept_len [B] (-1: a faulted request, left alone).  Tree node j was
    written at position committed + j.  Returns (new committed [B], status [B]).  The copies run
    in path order, one row (in every plane) at a time."""
    pool = np.asarray(pool)
    planes = pool if pool.ndim == 3 else pool[None]
    num_slots = planes.shape[1]
    B, N = np.asarray(accept_index).shape
    max_pos = np.asarray(slot_table).shape[1]
    new = np.array(committed, dtype=np.int64).copy()
    status = np.zeros(B, np.int32)
    for b in range(B):
        L = int(accept_len[b])
        c = int(committed[b])
        if L < 0:
            continue
        path = [int(accept_index[b][i]) for i in range(L + 1)] if L < N else []
        if c < 0 or c + N > max_pos or L >= N or any(a < 0 or a >= N for a in path):
            status[b] = KV_BAD_POSITION
            continue
        slots = [int(slot_table[b][c + a]) for a in path]
        dests = [int(slot_table[b][c + i]) for i in range(L + 1)]
        if any(s < 0 or s >= num_slots for s in slots + dests):
            status[b] = KV_BAD_SLOT
            continue
        for i in range(1, L + 1):
            src, dst = slots[i], dests[i]
            if src != dst:
                planes[:, dst] = planes[:, src].copy()
        new[b] = c + L + 1
    return new.astype(np.int32), status


# ---------------------------------------------------------------------------------------
# Adaptive verification budget ("The speculative decoding zoo", section "The finer loop:
# DSpark's confidence budget": every (request, position) slot scores the running product of the
# request's confidences up to it, a global top-k admits the best slots, ties go to the earlier
# position, and the budget maximises expected accepted tokens per unit of step cost;
# "Inference Systems Frontier: new models and speculative decoding", section "Deciding how much
# to verify by load": the same planner on a toy cost model).
# Readings: confidences are clamped to [0, 1] with NaN read as 0; survival is the running
# product in fp32 (the precision the GPU decides in); equal scores go to the earlier position,
# then the lower request index; slots past a request's number of drafts never compete; the
# gains are summed in fp64; cost[b] is the caller's cost of a step that admits b draft slots
# (drafting plus verifying B + b tokens); the first maximal rate wins.
# ---------------------------------------------------------------------------------------
BUDGET_MAX_SLOTS = 16384


def plan_budget(conf, cost, num_drafts=None):
    """conf [B, K] confidences; cost [B*K + 1]; num_drafts [B] or None (all K).
    Returns dict(budget, admitted [B], rate, boundary) where admitted[r] is the number of
    request r's leading slots admitted and boundary flags a maximal rate that another budget
    matches within 1e-12 (relative)."""
    c = np.nan_to_num(np.asarray(conf, np.float32), nan=0.0)
    c = np.clip(c, np.float32(0.0), np.float32(1.0))
    B, K = c.shape
    n_ok = np.full(B, K) if num_drafts is None else np.clip(np.asarray(num_drafts), 0, K)
    surv = np.empty((B, K), np.float32)
    run = np.ones(B, np.float32)
    for i in range(K):
        run = (run * c[:, i]).astype(np.float32)
        surv[:, i] = run
    slots = [(float(surv[r, i]), i, r) for r in range(B) for i in range(int(n_ok[r]))]
    slots.sort(key=lambda t: (-t[0], t[1], t[2]))
    gain = [0.0]
    for s, _, _ in slots:
        gain.append(gain[-1] + s)
    cost = np.asarray(cost, np.float64)
    rates = np.array([(B + gain[b]) / cost[b] for b in range(len(slots) + 1)])
    best = int(np.argmax(rates))
    others = np.delete(rates, best)
    boundary = bool(others.size and np.any(np.abs(others - rates[best]) <= 1e-12 * abs(rates[best])))
    admitted = np.zeros(B, np.int32)
    for _, i, r in slots[:best]:
        admitted[r] = max(admitted[r], i + 1)
    return dict(budget=best, admitted=admitted, rate=float(rates[best]), boundary=boundary)
