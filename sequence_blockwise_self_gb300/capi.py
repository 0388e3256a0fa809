"""ctypes binding of the C ABI in include/ring_attn.h.

Argument marshalling only: every step of the attention runs in the sm_103a
kernels of libring_attn.so.  There is no fallback: if the library is not
built, every call raises.  torch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

OK = 0
ERR_NULL = -1
ERR_SHAPE = -2
ERR_UNSUPPORTED = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5
ERR_DEVICE_TIMEOUT = -6

_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def load():
    """Load libring_attn.so (it must have been built; see build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (call sequence_blockwise_self_gb300.build.build())")
    lib = ctypes.CDLL(path)
    I, P, S = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    IP = ctypes.POINTER(ctypes.c_int)
    I32P = ctypes.POINTER(ctypes.c_int32)
    lib.ring_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P]
    lib.ring_attn_fwd.restype = I
    lib.ring_attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.ring_attn_bwd_workspace_size.restype = S
    lib.ring_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    lib.ring_attn_bwd.restype = I
    lib.ring_attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P]
    lib.ring_attn_bwd_noalloc.restype = I
    lib.ring_attn_strerror.argtypes = [I]
    lib.ring_attn_strerror.restype = ctypes.c_char_p
    lib.ring_attn_device_status.argtypes = [P, IP]
    lib.ring_attn_device_status.restype = I
    lib.ring_attn_release.argtypes = []
    lib.ring_attn_release.restype = None
    lib.ring_attn_owner_rank.argtypes = [I, I, I, I]
    lib.ring_attn_owner_rank.restype = I
    lib.ring_attn_selftest_bounded_wait.argtypes = [ctypes.c_uint, P]
    lib.ring_attn_selftest_bounded_wait.restype = I
    lib.ring_attn_profile_enable.argtypes = [I]
    lib.ring_attn_profile_enable.restype = I
    lib.ring_attn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
    lib.ring_attn_profile_read.restype = I
    for f in (lib.ring_attn_fwd_plan, lib.ring_attn_bwd_plan):
        f.argtypes = [I, I, I, IP, IP, I32P, I32P, I32P]
        f.restype = I
    lib.ring_attn_step_plan.argtypes = [I, I, I, I, I, I, IP, IP, I32P, I32P, I32P]
    lib.ring_attn_step_plan.restype = I
    lib.ring_attn_schedule_launches.argtypes = [I, I]
    lib.ring_attn_schedule_launches.restype = I
    lib.ring_attn_schedule_pair.argtypes = [I, I, I, I, IP, IP]
    lib.ring_attn_schedule_pair.restype = I
    lib.ring_attn_fwd_step.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P]
    lib.ring_attn_fwd_step.restype = I
    lib.ring_attn_fwd_step_accumulate.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P]
    lib.ring_attn_fwd_step_accumulate.restype = I
    lib.ring_attn_bwd_rank_workspace_size.argtypes = [I] * 8
    lib.ring_attn_bwd_rank_workspace_size.restype = S
    lib.ring_attn_bwd_rank_begin.argtypes = [P, P, P] + [I] * 8 + [P, S, P]
    lib.ring_attn_bwd_rank_begin.restype = I
    lib.ring_attn_bwd_rank_step.argtypes = [P] * 6 + [I] * 10 + [P, S, P]
    lib.ring_attn_bwd_rank_step.restype = I
    lib.ring_attn_bwd_rank_end.argtypes = [P] + [I] * 8 + [P, S, P]
    lib.ring_attn_bwd_rank_end.restype = I
    lib.ring_attn_grad_to_bf16.argtypes = [P, P, ctypes.c_longlong, ctypes.c_float, P]
    lib.ring_attn_grad_to_bf16.restype = I
    lib.ring_attn_bwd_rank_dq_offset.argtypes = [I] * 8
    lib.ring_attn_bwd_rank_dq_offset.restype = S
    lib.ring_attn_add_f32.argtypes = [P, P, ctypes.c_longlong, P]
    lib.ring_attn_add_f32.restype = I
    lib.ring_attn_merge.argtypes = [P, P, P, P, ctypes.c_longlong, I, P, P]
    lib.ring_attn_merge.restype = I
    lib.ring_attn_ring_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.ring_attn_ring_fwd_workspace_size.restype = S
    lib.ring_attn_ring_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, P, S, P]
    lib.ring_attn_ring_fwd.restype = I
    lib.ring_attn_ring_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.ring_attn_ring_bwd_workspace_size.restype = S
    lib.ring_attn_ring_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, S, P]
    lib.ring_attn_ring_bwd.restype = I
    lib.ring_attn_ulysses_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.ring_attn_ulysses_workspace_size.restype = S
    lib.ring_attn_ulysses_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    lib.ring_attn_ulysses_fwd.restype = I
    lib.ring_attn_ulysses_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    lib.ring_attn_ulysses_bwd.restype = I
    lib.ring_attn_usp_workspace_size.argtypes = [I] * 8
    lib.ring_attn_usp_workspace_size.restype = S
    lib.ring_attn_usp_fwd.argtypes = [P, P, P, P, P] + [I] * 8 + [P, S, P]
    lib.ring_attn_usp_fwd.restype = I
    lib.ring_attn_usp_bwd.argtypes = [P] * 9 + [I] * 8 + [P, S, P]
    lib.ring_attn_usp_bwd.restype = I
    lib.ring_attn_ffn_workspace_size.argtypes = [I, I, I]
    lib.ring_attn_ffn_workspace_size.restype = S
    lib.ring_attn_ffn_fwd.argtypes = [P, P, P, P, P, P, ctypes.c_longlong, I, I, I, P, S, P]
    lib.ring_attn_ffn_fwd.restype = I
    lib.ring_attn_ffn_bwd_workspace_size.argtypes = [I, I, I]
    lib.ring_attn_ffn_bwd_workspace_size.restype = S
    lib.ring_attn_ffn_bwd.argtypes = [P] * 10 + [ctypes.c_longlong, I, I, I, P, S, P]
    lib.ring_attn_ffn_bwd.restype = I
    lib.ring_attn_bpt_bwd_workspace_size.argtypes = [I] * 9
    lib.ring_attn_bpt_bwd_workspace_size.restype = S
    lib.ring_attn_bpt_bwd.argtypes = [P] * 16 + [I] * 9 + [P, S, P]
    lib.ring_attn_bpt_bwd.restype = I
    lib.ring_attn_bpt_workspace_size.argtypes = [I, I, I, I]
    lib.ring_attn_bpt_workspace_size.restype = S
    lib.ring_attn_bpt_fwd.argtypes = [P] * 10 + [I] * 9 + [P, S, P]
    lib.ring_attn_bpt_fwd.restype = I
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().ring_attn_strerror(int(status)).decode()


# ------------------------------------------------------------- host queries

def owner_rank(L: int, n_chunks: int, causal: bool, pos: int) -> int:
    return load().ring_attn_owner_rank(int(L), int(n_chunks), int(bool(causal)), int(pos))


def _plan(fn, L, n_chunks, causal):
    lib = load()
    nb, nr = ctypes.c_int(0), ctypes.c_int(0)
    rc = fn(int(L), int(n_chunks), int(bool(causal)), ctypes.byref(nb), ctypes.byref(nr), None, None, None)
    if rc != OK:
        raise RingAttnError(rc, "plan")
    order = np.zeros(nb.value, dtype=np.int32)
    offsets = np.zeros(nb.value + 1, dtype=np.int32)
    ranges = np.zeros(2 * nr.value, dtype=np.int32)
    p32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    rc = fn(int(L), int(n_chunks), int(bool(causal)), None, None, p32(order), p32(offsets), p32(ranges))
    if rc != OK:
        raise RingAttnError(rc, "plan")
    visits = [[(int(ranges[2 * r]), int(ranges[2 * r + 1])) for r in range(offsets[u], offsets[u + 1])]
              for u in range(nb.value)]
    return {"order": order, "offsets": offsets, "ranges": ranges, "visits": visits}


# Ring-mode schedules (RING_ATTN_SCHEDULE_* of include/ring_attn.h): the
# chunk map and the order of the blocks.
SCHEDULES = {"fold": 0, "striped": 1, "contiguous": 2, "dfa": 3}


def schedule_code(striped: bool = False, schedule=None) -> int:
    """The C ABI's schedule code: `schedule` by name, else fold or striped."""
    if schedule is None:
        return SCHEDULES["striped" if striped else "fold"]
    if striped and schedule != "striped":
        raise ValueError("striped contradicts the schedule")
    return SCHEDULES[schedule]


def schedule_launches(n_chunks: int, schedule="fold") -> int:
    rc = load().ring_attn_schedule_launches(int(n_chunks), schedule_code(schedule=schedule))
    if rc < 0:
        raise RingAttnError(rc, "ring_attn_schedule_launches")
    return rc


def schedule_pairs(n_chunks: int, schedule="fold"):
    """Per launch, the (worker, query chunk, key/value chunk) blocks of the
    schedule (idle workers left out)."""
    lib = load()
    code = schedule_code(schedule=schedule)
    out = []
    for t in range(schedule_launches(n_chunks, schedule)):
        launch = []
        for w in range(int(n_chunks)):
            a, b = ctypes.c_int(0), ctypes.c_int(0)
            rc = lib.ring_attn_schedule_pair(int(n_chunks), code, t, w, ctypes.byref(a), ctypes.byref(b))
            if rc < 0:
                raise RingAttnError(rc, "ring_attn_schedule_pair")
            if rc == 1:
                launch.append((w, a.value, b.value))
        out.append(launch)
    return out


def step_plan(L: int, n_chunks: int, causal: bool, step: int, rank: int, striped: bool = False, schedule=None):
    """Ring mode: per 256-row block of the query chunk of worker `rank`'s
    block at launch `step`, the key/value chunk's tile ranges it visits
    (chunk-local indices)."""
    fn = load().ring_attn_step_plan
    code = schedule_code(striped, schedule)
    return _plan(lambda L_, N_, c_, *rest: fn(L_, N_, c_, code, int(step), int(rank), *rest),
                 L, n_chunks, causal)


def fwd_plan(L: int, n_chunks: int, causal: bool):
    """Per 256-row query block: its key/value tile ranges in ring order."""
    return _plan(load().ring_attn_fwd_plan, L, n_chunks, causal)


def bwd_plan(L: int, n_chunks: int, causal: bool):
    """Per key/value tile: its query tile ranges in ring order."""
    return _plan(load().ring_attn_bwd_plan, L, n_chunks, causal)


# --------------------------------------------------------------- device calls

def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_tensor(t, name, dtype, shape):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def ring_attn_fwd(q, k, v, n_chunks: int, causal: bool, o=None, lse=None, stream=None):
    """softmax(q k^T / sqrt(d)) v by ring-ordered blocks; returns (o, lse)."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    _check_tensor(q, "q", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(k, "k", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(v, "v", torch.bfloat16, (B, Hkv, L, d))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    _check_tensor(o, "o", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    rc = load().ring_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, d, int(n_chunks),
                              int(bool(causal)), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_fwd")
    return o, lse


# ------------------------------------------------------------------ ring mode

def ring_attn_fwd_step(q_chunk, k_chunk, v_chunk, n_chunks: int, causal: bool, rank: int, src: int, o_s=None,
                       lse_s=None, stream=None, striped: bool = False, schedule=None):
    """One ring step of rank `rank` against the key/value chunk of rank `src`
    (chunks in chunk order, see include/ring_attn.h); returns the fp32
    partial result (o_s [B,Hq,C,d], lse_s [B,Hq,C])."""
    import torch
    B, Hq, C, d = q_chunk.shape
    Hkv = k_chunk.shape[1]
    _check_tensor(q_chunk, "q_chunk", torch.bfloat16, (B, Hq, C, d))
    _check_tensor(k_chunk, "k_chunk", torch.bfloat16, (B, Hkv, C, d))
    _check_tensor(v_chunk, "v_chunk", torch.bfloat16, (B, Hkv, C, d))
    o_s = torch.empty((B, Hq, C, d), dtype=torch.float32, device=q_chunk.device) if o_s is None else o_s
    lse_s = torch.empty((B, Hq, C), dtype=torch.float32, device=q_chunk.device) if lse_s is None else lse_s
    _check_tensor(o_s, "o_s", torch.float32, (B, Hq, C, d))
    _check_tensor(lse_s, "lse_s", torch.float32, (B, Hq, C))
    rc = load().ring_attn_fwd_step(_ptr(q_chunk), _ptr(k_chunk), _ptr(v_chunk), _ptr(o_s), _ptr(lse_s), B, Hq, Hkv,
                                   C * int(n_chunks), d, int(n_chunks), int(bool(causal)),
                                   schedule_code(striped, schedule), int(rank), int(src), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_fwd_step")
    return o_s, lse_s


def ring_attn_fwd_step_accumulate(q_chunk, k_chunk, v_chunk, o_run, lse_run, n_chunks: int, causal: bool, rank: int,
                                  src: int, stream=None, striped: bool = False, schedule=None):
    """The block of ring_attn_fwd_step (rank's queries, src's keys) merged
    in place into the running fp32 result (o_run [B,Hq,C,d], lse_run
    [B,Hq,C]; lse_run = -inf is the empty result).  Returns (o_run, lse_run)."""
    import torch
    B, Hq, C, d = q_chunk.shape
    Hkv = k_chunk.shape[1]
    _check_tensor(q_chunk, "q_chunk", torch.bfloat16, (B, Hq, C, d))
    _check_tensor(k_chunk, "k_chunk", torch.bfloat16, (B, Hkv, C, d))
    _check_tensor(v_chunk, "v_chunk", torch.bfloat16, (B, Hkv, C, d))
    _check_tensor(o_run, "o_run", torch.float32, (B, Hq, C, d))
    _check_tensor(lse_run, "lse_run", torch.float32, (B, Hq, C))
    rc = load().ring_attn_fwd_step_accumulate(_ptr(q_chunk), _ptr(k_chunk), _ptr(v_chunk), _ptr(o_run), _ptr(lse_run),
                                              B, Hq, Hkv, C * int(n_chunks), d, int(n_chunks), int(bool(causal)),
                                              schedule_code(striped, schedule), int(rank), int(src), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_fwd_step_accumulate")
    return o_run, lse_run


class RankBackward:
    """One rank's share of the ring-mode backward (ring_attn_bwd_rank_* of
    include/ring_attn.h) on its chunks [B, H, C, d] in chunk order: begin()
    forms the statistics, step() adds one block (the rank's queries against
    src's keys) into the rank's dQ and into the travelling fp32 dK/dV of
    src's chunk, end() returns dq."""

    def __init__(self, o_chunk, dO_chunk, lse_chunk, Hkv: int, n_chunks: int, causal: bool, striped: bool = False,
                 schedule=None, stream=None):
        import torch
        B, Hq, C, d = o_chunk.shape
        _check_tensor(o_chunk, "o_chunk", torch.bfloat16, (B, Hq, C, d))
        _check_tensor(dO_chunk, "dO_chunk", torch.bfloat16, (B, Hq, C, d))
        _check_tensor(lse_chunk, "lse_chunk", torch.float32, (B, Hq, C))
        self.shape = (B, Hq, int(Hkv), C * int(n_chunks), d, int(n_chunks), int(bool(causal)),
                      schedule_code(striped, schedule))
        nbytes = int(load().ring_attn_bwd_rank_workspace_size(*self.shape))
        if nbytes == 0:
            raise RingAttnError(ERR_SHAPE, "ring_attn_bwd_rank_workspace_size")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=o_chunk.device)
        self.dO = dO_chunk
        self.stream = stream
        rc = load().ring_attn_bwd_rank_begin(_ptr(o_chunk), _ptr(dO_chunk), _ptr(lse_chunk), *self.shape,
                                             _ptr(self.ws), nbytes, _stream(stream))
        if rc != OK:
            raise RingAttnError(rc, "ring_attn_bwd_rank_begin")

    def step(self, q_chunk, k_chunk, v_chunk, dk_acc, dv_acc, rank: int, src: int):
        import torch
        B, Hq, Hkv, L, d = self.shape[:5]
        C = L // self.shape[5]
        _check_tensor(q_chunk, "q_chunk", torch.bfloat16, (B, Hq, C, d))
        for t, n in ((k_chunk, "k_chunk"), (v_chunk, "v_chunk")):
            _check_tensor(t, n, torch.bfloat16, (B, Hkv, C, d))
        for t, n in ((dk_acc, "dk_acc"), (dv_acc, "dv_acc")):
            _check_tensor(t, n, torch.float32, (B, Hkv, C, d))
        rc = load().ring_attn_bwd_rank_step(_ptr(q_chunk), _ptr(k_chunk), _ptr(v_chunk), _ptr(self.dO), _ptr(dk_acc),
                                            _ptr(dv_acc), *self.shape, int(rank), int(src), _ptr(self.ws),
                                            self.ws.numel(), _stream(self.stream))
        if rc != OK:
            raise RingAttnError(rc, "ring_attn_bwd_rank_step")

    def dq_accumulator(self):
        """The rank's fp32 dQ accumulator (a view into the workspace, in the
        library's own order): what a DistFlashAttention helper sends back to
        the owner of the query chunk."""
        import torch
        off = int(load().ring_attn_bwd_rank_dq_offset(*self.shape))
        if off == 0:
            raise RingAttnError(ERR_SHAPE, "ring_attn_bwd_rank_dq_offset")
        B, Hq, C, d = self.dO.shape
        return self.ws[off:off + 4 * B * Hq * C * d].view(torch.float32)

    def add_dq(self, partial):
        """Add a helper's dQ accumulator (see dq_accumulator) into this rank's."""
        add_f32(self.dq_accumulator(), partial, stream=self.stream)

    def end(self, dq_chunk=None):
        import torch
        if dq_chunk is None:
            dq_chunk = torch.empty_like(self.dO)
        rc = load().ring_attn_bwd_rank_end(_ptr(dq_chunk), *self.shape, _ptr(self.ws), self.ws.numel(),
                                           _stream(self.stream))
        if rc != OK:
            raise RingAttnError(rc, "ring_attn_bwd_rank_end")
        return dq_chunk


def grad_to_bf16(acc, scale: float, out=None, stream=None):
    """bf16(scale * acc) for an fp32 accumulator (e.g. a travelling dK, dV)."""
    import torch
    if not isinstance(acc, torch.Tensor) or acc.dtype != torch.float32 or not acc.is_cuda or not acc.is_contiguous():
        raise TypeError("acc must be a contiguous fp32 CUDA tensor")
    out = torch.empty(acc.shape, dtype=torch.bfloat16, device=acc.device) if out is None else out
    rc = load().ring_attn_grad_to_bf16(_ptr(acc), _ptr(out), acc.numel(), float(scale), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_grad_to_bf16")
    return out


def add_f32(dst, src, stream=None):
    """In place: dst += src (contiguous fp32 CUDA tensors of equal size)."""
    import torch
    for t, n in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous fp32 CUDA tensor")
    if dst.numel() != src.numel():
        raise ValueError("dst and src differ in size")
    rc = load().ring_attn_add_f32(_ptr(dst), _ptr(src), dst.numel(), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_add_f32")
    return dst


def ring_attn_merge(o, lse, o_s, lse_s, o_out=None, stream=None):
    """In place: (o, lse) <- log-sum-exp merge of (o, lse) and (o_s, lse_s)
    (fp32, [..., d] and [...]); optionally bf16(o) into o_out.  Returns (o, lse)."""
    import torch
    d = o.shape[-1]
    rows = lse.numel()
    _check_tensor(o, "o", torch.float32, tuple(lse.shape) + (d,))
    _check_tensor(lse, "lse", torch.float32, tuple(lse.shape))
    _check_tensor(o_s, "o_s", torch.float32, tuple(o.shape))
    _check_tensor(lse_s, "lse_s", torch.float32, tuple(lse.shape))
    if o_out is not None:
        _check_tensor(o_out, "o_out", torch.bfloat16, tuple(o.shape))
    rc = load().ring_attn_merge(_ptr(o), _ptr(lse), _ptr(o_s), _ptr(lse_s), rows, d, _ptr(o_out), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_merge")
    return o, lse


def ring_fwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, striped: bool = False, schedule=None) -> int:
    return int(load().ring_attn_ring_fwd_workspace_size(B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)),
                                                         schedule_code(striped, schedule)))


def ring_attn_ring_fwd(q, k, v, n_chunks: int, causal: bool, o=None, lse=None, workspace=None, stream=None,
                       striped: bool = False, schedule=None):
    """The forward of ring_attn_fwd computed the ring-mode way (every rank's
    steps as separate launches, merged step by step); returns (o, lse)."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    _check_tensor(q, "q", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(k, "k", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(v, "v", torch.bfloat16, (B, Hkv, L, d))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(o, "o", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    ws_bytes = ring_fwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, striped, schedule)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    rc = load().ring_attn_ring_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, d, int(n_chunks),
                                   int(bool(causal)), schedule_code(striped, schedule), _ptr(workspace),
                                   int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ring_fwd")
    return o, lse


def ring_bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, striped: bool = False, schedule=None) -> int:
    return int(load().ring_attn_ring_bwd_workspace_size(B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)),
                                                         schedule_code(striped, schedule)))


def ring_attn_ring_bwd(q, k, v, o, lse, dO, n_chunks: int, causal: bool, dq=None, dk=None, dv=None, workspace=None,
                       stream=None, striped: bool = False, schedule=None):
    """The backward computed the ring-mode way (every rank's steps as
    separate launches); returns (dq, dk, dv)."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    for t, n, s in ((q, "q", (B, Hq, L, d)), (k, "k", (B, Hkv, L, d)), (v, "v", (B, Hkv, L, d)),
                    (o, "o", (B, Hq, L, d)), (dO, "dO", (B, Hq, L, d))):
        _check_tensor(t, n, torch.bfloat16, s)
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(ring_bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, striped, schedule), 1),
                                dtype=torch.uint8, device=q.device)
    rc = load().ring_attn_ring_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)),
                                   schedule_code(striped, schedule),
                                   _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                   _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ring_bwd")
    return dq, dk, dv


# ------------------------------------------------------------------ Ulysses

def ulysses_workspace_size(B, Hq, Hkv, L, d, n_ranks, causal) -> int:
    return int(load().ring_attn_ulysses_workspace_size(B, Hq, Hkv, L, d, int(n_ranks), int(bool(causal))))


def _ulysses_shapes(q, k):
    N, B, Hq, C, d = q.shape
    return N, B, Hq, k.shape[2], C * N, C, d


def ring_attn_ulysses_fwd(q, k, v, causal: bool, o=None, lse=None, workspace=None, stream=None):
    """Ulysses on one GPU: q [N,B,Hq,C,d], k, v [N,B,Hkv,C,d] (sequence
    shards, rank-major) -> (o [N,B,Hq,C,d], lse [N,B,Hq,C])."""
    import torch
    N, B, Hq, Hkv, L, C, d = _ulysses_shapes(q, k)
    _check_tensor(q, "q", torch.bfloat16, (N, B, Hq, C, d))
    _check_tensor(k, "k", torch.bfloat16, (N, B, Hkv, C, d))
    _check_tensor(v, "v", torch.bfloat16, (N, B, Hkv, C, d))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((N, B, Hq, C), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(o, "o", torch.bfloat16, (N, B, Hq, C, d))
    _check_tensor(lse, "lse", torch.float32, (N, B, Hq, C))
    if workspace is None:
        workspace = torch.empty(max(ulysses_workspace_size(B, Hq, Hkv, L, d, N, causal), 1), dtype=torch.uint8,
                                device=q.device)
    rc = load().ring_attn_ulysses_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, d, N,
                                      int(bool(causal)), _ptr(workspace),
                                      int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ulysses_fwd")
    return o, lse


def ring_attn_ulysses_bwd(q, k, v, o, lse, dO, causal: bool, dq=None, dk=None, dv=None, workspace=None,
                          stream=None):
    """Gradients for Ulysses on one GPU, all tensors as sequence shards
    (see ring_attn_ulysses_fwd); returns (dq, dk, dv)."""
    import torch
    N, B, Hq, Hkv, L, C, d = _ulysses_shapes(q, k)
    for t, n, s in ((q, "q", (N, B, Hq, C, d)), (k, "k", (N, B, Hkv, C, d)), (v, "v", (N, B, Hkv, C, d)),
                    (o, "o", (N, B, Hq, C, d)), (dO, "dO", (N, B, Hq, C, d))):
        _check_tensor(t, n, torch.bfloat16, s)
    _check_tensor(lse, "lse", torch.float32, (N, B, Hq, C))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(ulysses_workspace_size(B, Hq, Hkv, L, d, N, causal), 1), dtype=torch.uint8,
                                device=q.device)
    rc = load().ring_attn_ulysses_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                      _ptr(dv), B, Hq, Hkv, L, d, N, int(bool(causal)), _ptr(workspace),
                                      int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ulysses_bwd")
    return dq, dk, dv


def usp_workspace_size(B, Hq, Hkv, L, d, ulysses_degree, ring_degree, causal) -> int:
    return int(load().ring_attn_usp_workspace_size(int(B), int(Hq), int(Hkv), int(L), int(d), int(ulysses_degree),
                                                    int(ring_degree), int(bool(causal))))


def ring_attn_usp_fwd(q, k, v, ulysses_degree: int, causal: bool, o=None, lse=None, workspace=None, stream=None):
    """USP on one GPU: q [N,B,Hq,C,d], k, v [N,B,Hkv,C,d] as the N = U*R
    sequence shards stacked rank-major (rank r*U + u), U = ulysses_degree,
    R = N / U; returns (o [N,B,Hq,C,d], lse [N,B,Hq,C])."""
    import torch
    N, B, Hq, Hkv, L, C, d = _ulysses_shapes(q, k)
    U = int(ulysses_degree)
    if U <= 0 or N % U:
        raise ValueError("the shard count must be a multiple of the Ulysses degree")
    _check_tensor(q, "q", torch.bfloat16, (N, B, Hq, C, d))
    _check_tensor(k, "k", torch.bfloat16, (N, B, Hkv, C, d))
    _check_tensor(v, "v", torch.bfloat16, (N, B, Hkv, C, d))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((N, B, Hq, C), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(o, "o", torch.bfloat16, (N, B, Hq, C, d))
    _check_tensor(lse, "lse", torch.float32, (N, B, Hq, C))
    if workspace is None:
        workspace = torch.empty(max(usp_workspace_size(B, Hq, Hkv, L, d, U, N // U, causal), 1), dtype=torch.uint8,
                                device=q.device)
    rc = load().ring_attn_usp_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, d, U, N // U,
                                  int(bool(causal)), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                  _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_usp_fwd")
    return o, lse


def ring_attn_usp_bwd(q, k, v, o, lse, dO, ulysses_degree: int, causal: bool, dq=None, dk=None, dv=None,
                      workspace=None, stream=None):
    """Gradients for USP on one GPU, all tensors as sequence shards (see
    ring_attn_usp_fwd); returns (dq, dk, dv)."""
    import torch
    N, B, Hq, Hkv, L, C, d = _ulysses_shapes(q, k)
    U = int(ulysses_degree)
    if U <= 0 or N % U:
        raise ValueError("the shard count must be a multiple of the Ulysses degree")
    for t, n, sh in ((q, "q", (N, B, Hq, C, d)), (k, "k", (N, B, Hkv, C, d)), (v, "v", (N, B, Hkv, C, d)),
                     (o, "o", (N, B, Hq, C, d)), (dO, "dO", (N, B, Hq, C, d))):
        _check_tensor(t, n, torch.bfloat16, sh)
    _check_tensor(lse, "lse", torch.float32, (N, B, Hq, C))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(usp_workspace_size(B, Hq, Hkv, L, d, U, N // U, causal), 1), dtype=torch.uint8,
                                device=q.device)
    rc = load().ring_attn_usp_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, Hq, Hkv, L, d, U, N // U, int(bool(causal)), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_usp_bwd")
    return dq, dk, dv


def ffn_workspace_size(D: int, F: int, block_rows: int) -> int:
    return int(load().ring_attn_ffn_workspace_size(int(D), int(F), int(block_rows)))


def ring_attn_ffn_fwd(x, w1, b1, w2, b2, block_rows: int = 8192, y=None, workspace=None, stream=None):
    """Blockwise feed-forward: y = x + gelu(x W1^T + b1) W2^T + b2 row by row,
    block_rows rows at a time.  x [M, D] bf16; w1 [F, D], w2 [D, F] bf16
    (output-major, as a linear layer's weight); b1 [F], b2 [D] fp32.  y may
    be x (in place)."""
    import torch
    if x.dim() != 2 or w1.dim() != 2:
        raise ValueError("x must be [M, D] and w1 [F, D]")
    M, D = x.shape
    F = w1.shape[0]
    _check_tensor(x, "x", torch.bfloat16, (M, D))
    _check_tensor(w1, "w1", torch.bfloat16, (F, D))
    _check_tensor(w2, "w2", torch.bfloat16, (D, F))
    _check_tensor(b1, "b1", torch.float32, (F,))
    _check_tensor(b2, "b2", torch.float32, (D,))
    y = torch.empty_like(x) if y is None else y
    _check_tensor(y, "y", torch.bfloat16, (M, D))
    if workspace is None:
        workspace = torch.empty(max(ffn_workspace_size(D, F, block_rows), 1), dtype=torch.uint8, device=x.device)
    rc = load().ring_attn_ffn_fwd(_ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), _ptr(y), M, D, F,
                                  int(block_rows), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ffn_fwd")
    return y


def ffn_bwd_workspace_size(D: int, F: int, block_rows: int) -> int:
    return int(load().ring_attn_ffn_bwd_workspace_size(int(D), int(F), int(block_rows)))


def ring_attn_ffn_bwd(x, w1, b1, w2, dy, block_rows: int = 8192, workspace=None, stream=None, dx=None, dw1=None,
                      db1=None, dw2=None, db2=None):
    """Backward of ring_attn_ffn_fwd for the loss sum(dy * y): returns
    (dx [M, D] bf16, dw1 [F, D], db1 [F], dw2 [D, F], db2 [D] fp32); the
    outputs are allocated unless passed in."""
    import torch
    M, D = x.shape
    F = w1.shape[0]
    _check_tensor(x, "x", torch.bfloat16, (M, D))
    _check_tensor(w1, "w1", torch.bfloat16, (F, D))
    _check_tensor(w2, "w2", torch.bfloat16, (D, F))
    _check_tensor(b1, "b1", torch.float32, (F,))
    _check_tensor(dy, "dy", torch.bfloat16, (M, D))
    dev = x.device
    dx = torch.empty_like(x) if dx is None else dx
    dw1 = torch.empty((F, D), dtype=torch.float32, device=dev) if dw1 is None else dw1
    db1 = torch.empty((F,), dtype=torch.float32, device=dev) if db1 is None else db1
    dw2 = torch.empty((D, F), dtype=torch.float32, device=dev) if dw2 is None else dw2
    db2 = torch.empty((D,), dtype=torch.float32, device=dev) if db2 is None else db2
    _check_tensor(dx, "dx", torch.bfloat16, (M, D))
    for t, n, sh in ((dw1, "dw1", (F, D)), (db1, "db1", (F,)), (dw2, "dw2", (D, F)), (db2, "db2", (D,))):
        _check_tensor(t, n, torch.float32, sh)
    if workspace is None:
        workspace = torch.empty(max(ffn_bwd_workspace_size(D, F, block_rows), 1), dtype=torch.uint8, device=dev)
    rc = load().ring_attn_ffn_bwd(_ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(dy), _ptr(dx), _ptr(dw1), _ptr(db1),
                                  _ptr(dw2), _ptr(db2), M, D, F, int(block_rows), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_ffn_bwd")
    return dx, dw1, db1, dw2, db2


def bpt_workspace_size(Hq: int, d: int, F: int, block_rows: int) -> int:
    return int(load().ring_attn_bpt_workspace_size(int(Hq), int(d), int(F), int(block_rows)))


def ring_attn_bpt_fwd(q, k, v, w1, b1, w2, b2, n_chunks: int, causal: bool, block_rows: int = 8192, a_tok=None,
                      lse=None, y=None, workspace=None, stream=None):
    """Blockwise transformer forward: per block of query rows, the block's
    attention (written token-major, a_tok [B, L, Hq*d]) and then
    y = a_tok + gelu(a_tok W1^T + b1) W2^T + b2 on its rows.  q [B,Hq,L,d],
    k, v [B,Hkv,L,d] bf16; w1 [F, Hq*d], w2 [Hq*d, F] bf16; b1, b2 fp32.
    Returns (a_tok, lse, y)."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    D, F = Hq * d, w1.shape[0]
    _check_tensor(q, "q", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(k, "k", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(v, "v", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(w1, "w1", torch.bfloat16, (F, D))
    _check_tensor(w2, "w2", torch.bfloat16, (D, F))
    _check_tensor(b1, "b1", torch.float32, (F,))
    _check_tensor(b2, "b2", torch.float32, (D,))
    a_tok = torch.empty((B, L, D), dtype=torch.bfloat16, device=q.device) if a_tok is None else a_tok
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device) if lse is None else lse
    y = torch.empty((B, L, D), dtype=torch.bfloat16, device=q.device) if y is None else y
    _check_tensor(a_tok, "a_tok", torch.bfloat16, (B, L, D))
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    _check_tensor(y, "y", torch.bfloat16, (B, L, D))
    if workspace is None:
        workspace = torch.empty(max(bpt_workspace_size(Hq, d, F, block_rows), 1), dtype=torch.uint8,
                                device=q.device)
    rc = load().ring_attn_bpt_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a_tok), _ptr(lse), _ptr(w1), _ptr(b1), _ptr(w2),
                                  _ptr(b2), _ptr(y), B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)), F,
                                  int(block_rows), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                  _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_bpt_fwd")
    return a_tok, lse, y


def bpt_bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, F, block_rows) -> int:
    return int(load().ring_attn_bpt_bwd_workspace_size(int(B), int(Hq), int(Hkv), int(L), int(d), int(n_chunks),
                                                        int(bool(causal)), int(F), int(block_rows)))


def ring_attn_bpt_bwd(q, k, v, a_tok, lse, w1, b1, w2, dy, n_chunks: int, causal: bool, block_rows: int = 8192,
                      workspace=None, stream=None, outs=None):
    """Backward of ring_attn_bpt_fwd for the loss sum(dy * y), dy [B, L, Hq*d]
    bf16: returns (dq, dk, dv, dw1, db1, dw2, db2), allocated unless `outs`
    passes all seven."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    D, F = Hq * d, w1.shape[0]
    _check_tensor(q, "q", torch.bfloat16, (B, Hq, L, d))
    _check_tensor(k, "k", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(v, "v", torch.bfloat16, (B, Hkv, L, d))
    _check_tensor(a_tok, "a_tok", torch.bfloat16, (B, L, D))
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    _check_tensor(w1, "w1", torch.bfloat16, (F, D))
    _check_tensor(w2, "w2", torch.bfloat16, (D, F))
    _check_tensor(b1, "b1", torch.float32, (F,))
    _check_tensor(dy, "dy", torch.bfloat16, (B, L, D))
    dev = q.device
    if outs is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dw1 = torch.empty((F, D), dtype=torch.float32, device=dev)
        db1 = torch.empty((F,), dtype=torch.float32, device=dev)
        dw2 = torch.empty((D, F), dtype=torch.float32, device=dev)
        db2 = torch.empty((D,), dtype=torch.float32, device=dev)
    else:
        dq, dk, dv, dw1, db1, dw2, db2 = outs
    for t, n, sh in ((dq, "dq", (B, Hq, L, d)), (dk, "dk", (B, Hkv, L, d)), (dv, "dv", (B, Hkv, L, d))):
        _check_tensor(t, n, torch.bfloat16, sh)
    for t, n, sh in ((dw1, "dw1", (F, D)), (db1, "db1", (F,)), (dw2, "dw2", (D, F)), (db2, "db2", (D,))):
        _check_tensor(t, n, torch.float32, sh)
    if workspace is None:
        workspace = torch.empty(max(bpt_bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal, F, block_rows), 1),
                                dtype=torch.uint8, device=dev)
    rc = load().ring_attn_bpt_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a_tok), _ptr(lse), _ptr(w1), _ptr(b1), _ptr(w2),
                                  _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dw1), _ptr(db1), _ptr(dw2), _ptr(db2),
                                  B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)), F, int(block_rows),
                                  _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_bpt_bwd")
    return dq, dk, dv, dw1, db1, dw2, db2


def bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal) -> int:
    return int(load().ring_attn_bwd_workspace_size(B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal))))


def ring_attn_bwd(q, k, v, o, lse, dO, n_chunks: int, causal: bool, dq=None, dk=None, dv=None, workspace=None,
                  stream=None):
    """Gradients of sum(dO * o) with respect to q, k, v; returns (dq, dk, dv)."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    for t, n, s in ((q, "q", (B, Hq, L, d)), (k, "k", (B, Hkv, L, d)), (v, "v", (B, Hkv, L, d)),
                    (o, "o", (B, Hq, L, d)), (dO, "dO", (B, Hq, L, d))):
        _check_tensor(t, n, torch.bfloat16, s)
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = bwd_workspace_size(B, Hq, Hkv, L, d, n_chunks, causal)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    rc = load().ring_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                              _ptr(dv), B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)), _ptr(workspace),
                              int(workspace.numel() * workspace.element_size()), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_bwd")
    return dq, dk, dv


def ring_attn_bwd_noalloc(q, k, v, o, lse, dO, n_chunks: int, causal: bool, dq, dk, dv, stream=None):
    """ring_attn_bwd for callers that cannot allocate device memory: the
    library works in its own static device array (see include/ring_attn.h)
    instead of a workspace.  dq, dk, dv must be passed in (allocated by the
    caller's own means); returns them."""
    import torch
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    for t, n, s in ((q, "q", (B, Hq, L, d)), (k, "k", (B, Hkv, L, d)), (v, "v", (B, Hkv, L, d)),
                    (o, "o", (B, Hq, L, d)), (dO, "dO", (B, Hq, L, d)), (dq, "dq", (B, Hq, L, d)),
                    (dk, "dk", (B, Hkv, L, d)), (dv, "dv", (B, Hkv, L, d))):
        _check_tensor(t, n, torch.bfloat16, s)
    _check_tensor(lse, "lse", torch.float32, (B, Hq, L))
    rc = load().ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                      _ptr(dv), B, Hq, Hkv, L, d, int(n_chunks), int(bool(causal)), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_bwd_noalloc")
    return dq, dk, dv


def selftest_bounded_wait(timeout_us: int, stream=None):
    """Launch the failure-detection self-test (a wait that can only time out)."""
    rc = load().ring_attn_selftest_bounded_wait(int(timeout_us), _stream(stream))
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_selftest_bounded_wait")


def device_status(stream=None):
    """Synchronise and return (status, site) of the device status word."""
    site = ctypes.c_int(0)
    rc = load().ring_attn_device_status(_stream(stream), ctypes.byref(site))
    return rc, site.value


KERNEL_NAMES = ("fwd", "bwd_pre", "bwd_main", "bwd_post", "ring_step", "ring_merge", "ring_io", "ulysses_a2a",
                "ffn_gemm")


def profile_enable(on: bool = True):
    load().ring_attn_profile_enable(int(bool(on)))


def profile_read():
    """{kernel: (summed ms, launches)} since the last read (waits for them)."""
    ms = (ctypes.c_double * len(KERNEL_NAMES))()   # RING_ATTN_N_KERNELS entries
    n = (ctypes.c_longlong * len(KERNEL_NAMES))()
    rc = load().ring_attn_profile_read(ms, n)
    if rc != OK:
        raise RingAttnError(rc, "ring_attn_profile_read")
    return {k: (ms[i], int(n[i])) for i, k in enumerate(KERNEL_NAMES)}


def release():
    load().ring_attn_release()
