"""Python face of the fp64 oracle (ctypes over ring_attn_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's
CPU-baseline leg may call it.

Citations name the web page "Large-scale distributed AI model training
series: sequence parallelism" (the "SP series") and its sections:
  * section 2.3 (Ring Self-Attention): attention is Q K^T then Score V; each
    of N devices holds L/N tokens and the key/value blocks travel round a
    ring, N-1 transfers and N block computations per device;
  * section 6.2 (Ring Attention): one ring carries K and V together and the
    per-step partial results are merged with the online-softmax correction;
  * section 7.2 (DistFlashAttention): with contiguous causal chunks the
    ring is unbalanced; a worker that would wait takes over blocks of a
    later worker (8 steps become 5 in the pages' example);
  * section 8.2 (USP): for a causal model the sequence is split by folding
    it, so that every device gets the same amount of work.

Inputs are numpy float64 arrays holding the bf16 values (the caller widens
them); layout q/o/dO [B,Hq,L,d], k/v [B,Hkv,L,d], lse [B,Hq,L].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/liboracle.so (plain gcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    I = ctypes.c_int
    lib.oracle_fwd.argtypes = [_dp, _dp, _dp, I, I, I, I, I, I, _dp, _dp, I]
    lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, I, I, I, I, I, I, _ip, I, _dp, _dp, I]
    lib.oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, I, I, I, I, I, I, _dp, _dp, _dp, _dp, _dp, I]
    lib.oracle_bwd_rows.argtypes = [_dp, _dp, _dp, _dp, I, I, I, I, I, I, _ip, I, _ip, I,
                                    _dp, _dp, _dp, I]
    lib.oracle_ring_fwd.argtypes = [_dp, _dp, _dp, I, I, I, I, I, I, I, I, _dp, _dp, I]
    lib.oracle_ring_step.argtypes = [_dp, _dp, _dp, I, I, I, I, I, I, I, I, I, I, _dp, _dp, I]
    lib.oracle_ring_step_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp] + [I] * 10 + [_dp, _dp, _dp, I]
    lib.oracle_ring_step_bwd.restype = ctypes.c_int
    lib.oracle_merge.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, I]
    lib.oracle_merge.restype = None
    lib.oracle_owner_rank.argtypes = [I, I, I, I, I]
    lib.oracle_ffn.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, I, I, _dp, _dp, I]
    lib.oracle_ffn.restype = ctypes.c_int
    lib.oracle_ffn_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, I, I, _dp, _dp, _dp, _dp, _dp, _dp, _dp, I]
    lib.oracle_ffn_bwd.restype = ctypes.c_int
    for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_bwd, lib.oracle_bwd_rows,
              lib.oracle_ring_fwd, lib.oracle_ring_step, lib.oracle_owner_rank):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _swap_library(path):
    """Point this module at another build of the oracle source (used by the
    mutation test, which plants mistakes in a copy); returns the previous
    handle so the caller can restore it."""
    global _lib
    prev = _lib
    _lib = _bind(ctypes.CDLL(path)) if path else None
    return prev


def _restore_library(handle):
    global _lib
    _lib = handle


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _shape(q, k):
    B, Hq, L, d = q.shape
    Bk, Hkv, Lk, dk = k.shape
    if (B, L, d) != (Bk, Lk, dk) or Hq % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape}")
    return B, Hq, Hkv, L, d


def _threads(n):
    if n:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _check(rc):
    if rc < 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return rc


def fwd(q, k, v, causal: bool, threads: int = 0):
    """Plain definition of softmax(Q K^T / sqrt(d)) V (SP series section 2.3).

    Returns (o [B,Hq,L,d], lse [B,Hq,L]); lse is the natural log-sum-exp of
    the scaled scores."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, L, d = _shape(q, k)
    o = np.zeros((B, Hq, L, d))
    lse = np.zeros((B, Hq, L))
    _check(_load().oracle_fwd(_p(q), _p(k), _p(v), B, Hq, Hkv, L, d, int(causal), _p(o), _p(lse),
                              _threads(threads)))
    return o, lse


def fwd_rows(q, k, v, causal: bool, rows, threads: int = 0):
    """The plain definition on selected query rows (same rows for every head).

    Returns (o_rows [B,Hq,R,d], lse_rows [B,Hq,R]) and the thread count used."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, L, d = _shape(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    R = rows.size
    o = np.zeros((B, Hq, R, d))
    lse = np.zeros((B, Hq, R))
    nt = _check(_load().oracle_fwd_rows(_p(q), _p(k), _p(v), B, Hq, Hkv, L, d, int(causal),
                                        rows.ctypes.data_as(_ip), R, _p(o), _p(lse),
                                        _threads(threads)))
    return o, lse, nt


def bwd(q, k, v, dO, causal: bool, threads: int = 0):
    """Hand-derived backward of l = sum(dO * O).

    Returns (dq, dk, dv, lse, D) in fp64; D_i = dO_i . o_i."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, L, d = _shape(q, k)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    lse = np.zeros((B, Hq, L))
    D = np.zeros((B, Hq, L))
    _check(_load().oracle_bwd(_p(q), _p(k), _p(v), _p(dO), B, Hq, Hkv, L, d, int(causal), _p(dq),
                              _p(dk), _p(dv), _p(lse), _p(D), _threads(threads)))
    return dq, dk, dv, lse, D


def bwd_rows(q, k, v, dO, causal: bool, q_rows, k_rows, threads: int = 0):
    """Backward on sampled rows: dq on q_rows, dk/dv on k_rows.

    Returns (dq_rows [B,Hq,Rq,d], dk_rows [B,Hkv,Rk,d], dv_rows [B,Hkv,Rk,d])."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, L, d = _shape(q, k)
    qr = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int32))
    kr = np.ascontiguousarray(np.asarray(k_rows, dtype=np.int32))
    dq = np.zeros((B, Hq, qr.size, d))
    dk = np.zeros((B, Hkv, kr.size, d))
    dv = np.zeros((B, Hkv, kr.size, d))
    _check(_load().oracle_bwd_rows(_p(q), _p(k), _p(v), _p(dO), B, Hq, Hkv, L, d, int(causal),
                                   qr.ctypes.data_as(_ip), qr.size, kr.ctypes.data_as(_ip), kr.size,
                                   _p(dq), _p(dk), _p(dv), _threads(threads)))
    return dq, dk, dv


# Ring schedules (the oracle's SCHED_* codes): the chunk map and the order
# of the blocks.  "fold": contiguous chunks (encoder) or the folded
# sub-chunks {r, 2N-1-r} (causal, SP series section 8.2), N ring steps;
# "striped": rank r owns positions r, r+N, ...; "contiguous": causal with
# contiguous chunks, the plain (unbalanced) ring; "dfa": causal with
# contiguous chunks in DistFlashAttention's balanced schedule (section 7.2,
# see dfa_schedule).
SCHEDULES = {"fold": 0, "striped": 1, "contiguous": 2, "dfa": 3}


def _schedule(striped, schedule):
    if schedule is None:
        return SCHEDULES["striped" if striped else "fold"]
    if striped and schedule != "striped":
        raise ValueError("striped contradicts the schedule")
    return SCHEDULES[schedule]


def ring_fwd(q, k, v, causal: bool, n_chunks: int, threads: int = 0, striped: bool = False, schedule=None):
    """Ring form: per ring step partial (o_s, lse_s) merged by log-sum-exp
    (SP series sections 2.3 and 6.2; causal ranks own folded sub-chunks,
    section 8.2, or, with striped, the positions r, r+N, r+2N, ...; or
    contiguous chunks in ring order or DistFlashAttention's order, section
    7.2, with schedule="contiguous" / "dfa")."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, L, d = _shape(q, k)
    o = np.zeros((B, Hq, L, d))
    lse = np.zeros((B, Hq, L))
    _check(_load().oracle_ring_fwd(_p(q), _p(k), _p(v), B, Hq, Hkv, L, d, int(causal), int(n_chunks),
                                   _schedule(striped, schedule), _p(o), _p(lse), _threads(threads)))
    return o, lse


def ring_step(q, k, v, causal: bool, n_chunks: int, rank: int, src: int, threads: int = 0, striped: bool = False,
              schedule=None):
    """One ring step in isolation (SP series sections 2.3 and 6.2): the
    partial result (o_s, lse_s) of rank `rank`'s query rows against the keys
    and values of rank `src`.  Returned in global row order, [B,Hq,L,d] and
    [B,Hq,L]; rows of other ranks are 0 and -inf, as are rows of `rank` that
    see none of src's keys.  striped: rank r owns positions r, r+N, ...;
    schedule "contiguous" or "dfa": contiguous causal chunks."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, L, d = _shape(q, k)
    o = np.zeros((B, Hq, L, d))
    lse = np.full((B, Hq, L), -np.inf)
    _check(_load().oracle_ring_step(_p(q), _p(k), _p(v), B, Hq, Hkv, L, d, int(causal), int(n_chunks),
                                    int(rank), int(src), _schedule(striped, schedule), _p(o), _p(lse),
                                    _threads(threads)))
    return o, lse


def ring_step_bwd(q, k, v, dO, lse, D, causal: bool, n_chunks: int, rank: int, src: int, threads: int = 0,
                  striped: bool = False, schedule=None):
    """One ring block of the backward (SP series section 6.2): the
    contribution of rank's query rows against src's keys, with the full
    statistics lse, D [B,Hq,L] of the plain definition (oracle.bwd returns
    them): dq on rank's rows, dk and dv on src's rows (global row order,
    zero elsewhere).  Summed over every block: the plain backward."""
    q, k, v, dO, lse, D = (_f64(a) for a in (q, k, v, dO, lse, D))
    B, Hq, Hkv, L, d = _shape(q, k)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _check(_load().oracle_ring_step_bwd(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(D), B, Hq, Hkv, L, d, int(causal),
                                        int(n_chunks), int(rank), int(src), _schedule(striped, schedule), _p(dq),
                                        _p(dk), _p(dv), _threads(threads)))
    return dq, dk, dv


def merge(o_a, lse_a, o_b, lse_b):
    """Log-sum-exp merge of two partial results of the same rows (SP series
    section 6.2): returns (o, lse) with lse = log(e^lse_a + e^lse_b) and
    o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b; a side with lse = -inf
    contributes nothing."""
    o = np.array(o_a, dtype=np.float64, copy=True, order="C")
    lse = np.array(lse_a, dtype=np.float64, copy=True, order="C")
    ob = _f64(o_b)
    lb = _f64(lse_b)
    d = o.shape[-1]
    if ob.shape != o.shape or lb.shape != lse.shape or o.shape[:-1] != lse.shape:
        raise ValueError("merge: shape mismatch")
    _load().oracle_merge(_p(o), _p(lse), _p(ob), _p(lb), int(lse.size), int(d))
    return o, lse


def ffn(x, w1, b1, w2, b2, threads: int = 0, rows=None, hidden: bool = False):
    """The BPT feed-forward block with its residual (SP series section 4.2,
    two linear layers with a 4x up-projection, section 8):
    y = x + gelu(x W1 + b1) W2 + b2 with the exact GELU x Phi(x); x [M, D],
    W1 [D, F], W2 [F, D].  Rows are independent (blockwise order is moot).
    rows: optional row indices; then only those rows are computed and the
    result is y[rows] ([len(rows), D]).  hidden=True also returns the
    hidden activation gelu(x W1 + b1) of the same rows."""
    x, w1, b1, w2, b2 = (_f64(a) for a in (x, w1, b1, w2, b2))
    M, D = x.shape
    F = w1.shape[1]
    if w1.shape != (D, F) or w2.shape != (F, D) or b1.shape != (F,) or b2.shape != (D,):
        raise ValueError("ffn: shape mismatch")
    if rows is None:
        y = np.zeros((M, D))
        h = np.zeros((M, F)) if hidden else None
        _check(_load().oracle_ffn(_p(x), _p(w1), _p(b1), _p(w2), _p(b2), M, D, F, _p(y),
                                  _p(h) if hidden else None, _threads(threads)))
        return (y, h) if hidden else y
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    xs = np.ascontiguousarray(x[idx])
    n = idx.size
    y = np.zeros((n, D))
    h = np.zeros((n, F)) if hidden else None
    _check(_load().oracle_ffn(_p(xs), _p(w1), _p(b1), _p(w2), _p(b2), n, D, F, _p(y),
                              _p(h) if hidden else None, _threads(threads)))
    return (y, h) if hidden else y


def ffn_bwd(x, w1, b1, w2, dy, threads: int = 0, hidden: bool = False):
    """Gradients of sum(dy * y) for the FFN block of ffn() (the BPT section's
    backward, recomputing the block's hidden activation): returns dx [M, D],
    dW1 [D, F], db1 [F], dW2 [F, D], db2 [D] (oracle layout, W1 [D, F], W2
    [F, D]), by the chain rule with gelu'(a) = Phi(a) + a phi(a).
    hidden=True also returns h and da [M, F]."""
    x, w1, b1, w2, dy = (_f64(a) for a in (x, w1, b1, w2, dy))
    M, D = x.shape
    F = w1.shape[1]
    if w1.shape != (D, F) or w2.shape != (F, D) or b1.shape != (F,) or dy.shape != (M, D):
        raise ValueError("ffn_bwd: shape mismatch")
    dx, dw1, db1, dw2, db2 = np.zeros((M, D)), np.zeros((D, F)), np.zeros(F), np.zeros((F, D)), np.zeros(D)
    h = np.zeros((M, F)) if hidden else None
    da = np.zeros((M, F)) if hidden else None
    _check(_load().oracle_ffn_bwd(_p(x), _p(w1), _p(b1), _p(w2), _p(dy), M, D, F, _p(dx), _p(dw1), _p(db1), _p(dw2),
                                  _p(db2), _p(h) if hidden else None, _p(da) if hidden else None, _threads(threads)))
    return (dx, dw1, db1, dw2, db2, h, da) if hidden else (dx, dw1, db1, dw2, db2)


# ------------------------------------------------------------ chunk map (host)

def owner_rank(L: int, n_chunks: int, causal: bool, p: int, striped: bool = False, schedule=None) -> int:
    """Rank owning sequence position p: chunk p // (L/N) for the encoder
    and the contiguous causal schedules; for the causal fold the pair
    {r, 2N-1-r} of sub-chunks of length L/(2N) (SP series section 8.2);
    p mod N when striped."""
    r = _load().oracle_owner_rank(int(L), int(n_chunks), int(causal), _schedule(striped, schedule), int(p))
    if r < 0:
        raise ValueError("bad chunk map arguments")
    return r


def dfa_schedule(n_chunks: int):
    """DistFlashAttention's balanced causal schedule (SP series section 7.2:
    a worker that would wait in the plain ring takes over a later worker's
    block).  Returns one list per launch t = 0..N//2 of (worker, query
    chunk, key/value chunk): worker w >= t does its own block (w, w - t);
    worker w < t the block (N - t + w, w) of ring step N - t, unless that
    step is this launch (N even, t = N/2), when it stays idle."""
    N = int(n_chunks)
    out = []
    for t in range(N // 2 + 1):
        launch = []
        for w in range(N):
            if w >= t:
                launch.append((w, w, w - t))
            elif t < N - t:
                launch.append((w, N - t + w, w))
        out.append(launch)
    return out


def ring_sources(r: int, n_chunks: int):
    """Ring visiting order of rank r: at step s it holds the key/value block of
    rank (r - s) mod N, starting with its own (SP series section 2.3)."""
    return [(r - s) % n_chunks for s in range(n_chunks)]


def visible_pairs(L: int, causal: bool, tile: int):
    """Set of (query tile, key tile) pairs that hold at least one visible
    (i, j) position: all pairs for the encoder, key tile <= query tile for a
    causal model (position j <= i)."""
    nt = (L + tile - 1) // tile
    out = set()
    for a in range(nt):
        for b in range(nt):
            if not causal or b * tile <= min((a + 1) * tile, L) - 1:
                out.add((a, b))
    return out
