"""fp64 CPU oracle of the speculative-sampling verify step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` import this
package. The CUDA library never imports, links or calls it, and it imports nothing from the CUDA
library: the two share only the seeded input generator, which holds none of the method's
arithmetic.

``verify_ref.c`` is the oracle itself (plain C, fp64, its own Philox4x32-10). This module compiles it
with gcc on first use and wraps it with ctypes. ``brute.py`` holds the exact rational enumeration
that pins the oracle's joint output law.

Parity unpinned: the inverse-CDF tail rule (no crossing through rounding -> last positive weight),
the S == 0 residual fallback and the handling of -inf weights are conventions no page fixes; they
are covered by unit cases only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``verify_ref.c`` into ``liboracle.so`` (plain gcc, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Debug(ctypes.Structure):
    _fields_ = [("row_lse", ctypes.c_void_p), ("row_argmax", ctypes.c_void_p),
                ("p_x", ctypes.c_void_p), ("q_x", ctypes.c_void_p),
                ("seq_mass", ctypes.c_void_p), ("seq_fallback", ctypes.c_void_p), ("beta", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_philox4x32_10.restype = None
            L.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                         ctypes.c_uint32, ctypes.c_uint32]
            L.oracle_uniform.restype = ctypes.c_double
            L.oracle_verify_probs.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32] * 2 + \
                [ctypes.c_void_p] * 5
            L.oracle_verify_probs.restype = ctypes.c_int32
            L.oracle_verify.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.POINTER(_Debug), ctypes.c_int]
            L.oracle_verify.restype = ctypes.c_uint32
            L.oracle_verify_range.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.POINTER(_Debug), ctypes.c_int]
            L.oracle_verify_range.restype = ctypes.c_uint32
            L.oracle_verify_steps.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            L.oracle_verify_steps.restype = ctypes.c_uint32
            L.oracle_draw_bracket.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_draw_bracket.restype = ctypes.c_int32
            L.oracle_tree_probs.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32] * 2 + [ctypes.c_void_p] * 4
            L.oracle_tree_probs.restype = ctypes.c_int32
            L.oracle_verify_tree.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 4 + \
                [ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64] + \
                [ctypes.c_void_p] * 3
            L.oracle_verify_tree.restype = ctypes.c_uint32
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, step: int, seq: int, slot: int, purpose: int) -> float:
    return lib().oracle_uniform(seed, step, seq, slot, purpose)


def verify_probs(p, q, x, u_acc, u_smp):
    """Core rule on fp64 probabilities for one sequence.

    p: [gamma+1, V], q: [gamma, V], x: [gamma] draft tokens, u_acc: [gamma], u_smp: [gamma+1].
    Returns (n, tokens[gamma+1], S, fallback).
    """
    p = np.ascontiguousarray(p, dtype=np.float64)
    g = p.shape[0] - 1
    V = p.shape[1]
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(g, V) if g > 0 else np.zeros((1, V))
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(g) if g > 0 else np.zeros(1, np.int32)
    ua = np.ascontiguousarray(u_acc, dtype=np.float64).reshape(g) if g > 0 else np.zeros(1)
    us = np.ascontiguousarray(u_smp, dtype=np.float64).reshape(g + 1)
    out = np.zeros(g + 1, dtype=np.int32)
    S = np.zeros(1)
    fb = np.zeros(1, dtype=np.int32)
    n = lib().oracle_verify_probs(_ptr(p), _ptr(q), _ptr(x), g, V, _ptr(ua), _ptr(us), _ptr(out),
                                  _ptr(S), _ptr(fb))
    return n, out, float(S[0]), bool(fb[0])


class Result:
    def __init__(self, B, R_t, R_d):
        self.tokens = np.full(R_t, -7, dtype=np.int32)
        self.num_accepted = np.full(B, -7, dtype=np.int32)
        self.row_lse = np.full(R_t + R_d, np.nan)
        self.row_argmax = np.full(R_t, -7, dtype=np.int32)
        self.p_x = np.full(R_d, np.nan)
        self.q_x = np.full(R_d, np.nan)
        self.seq_mass = np.full(B, np.nan)
        self.seq_fallback = np.zeros(B, dtype=np.int32)
        self.beta = np.full(R_d, np.nan)
        self.status = 0


def verify(target, draft, draft_tokens, seq_offsets, gammas, V, temperature, seed, step,
           nthreads: int | None = None, seq_base: int = 0) -> Result:
    """Verify a CSR-packed batch on host arrays.

    target/draft: numpy arrays of float32 logits, or uint16 arrays holding raw bf16 bits, with
    shapes [R_t, V] / [R_d, V]. draft None with temperature > 0: the drafts are point masses (an
    n-gram drafter's). seq_base: the global index of sequence 0 when the batch is a contiguous range
    of a larger one (its uniforms are then the larger batch's). Returns a ``Result`` with tokens,
    counts and debug values.
    """
    target = np.ascontiguousarray(target)
    dtype = BF16 if target.dtype == np.uint16 else F32
    if dtype == F32:
        target = target.astype(np.float32, copy=False)
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        draft = draft.astype(np.uint16 if dtype == BF16 else np.float32, copy=False)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    gam = np.ascontiguousarray(gammas, dtype=np.int32)
    tok = None if draft_tokens is None else np.ascontiguousarray(draft_tokens, dtype=np.int32)
    B = len(gam)
    R_d = int(offs[-1]) if B else 0
    R_t = R_d + B
    res = Result(B, R_t, R_d)
    dbg = _Debug(_ptr(res.row_lse), _ptr(res.row_argmax), _ptr(res.p_x), _ptr(res.q_x),
                 _ptr(res.seq_mass), _ptr(res.seq_fallback), _ptr(res.beta))
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    res.status = lib().oracle_verify_range(_ptr(target), _ptr(draft), dtype, _ptr(tok), _ptr(offs),
                                           _ptr(gam), B, V, float(temperature), seed, step, int(seq_base),
                                           _ptr(res.tokens), _ptr(res.num_accepted), ctypes.byref(dbg),
                                           int(nthreads))
    return res


def verify_steps(target, draft, draft_tokens, seq_offsets, gammas, V, temperature, seed, step0, nsteps,
                 nthreads: int | None = None):
    """``verify`` for steps step0 .. step0 + nsteps - 1 of one batch (temperature > 0), each sequence's
    probabilities computed once (see ``oracle_verify_steps``). Returns (tokens [nsteps, R_t],
    num_accepted [nsteps, B], status)."""
    target = np.ascontiguousarray(target)
    dtype = BF16 if target.dtype == np.uint16 else F32
    if dtype == F32:
        target = target.astype(np.float32, copy=False)
    if draft is not None:
        draft = np.ascontiguousarray(draft).astype(np.uint16 if dtype == BF16 else np.float32, copy=False)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    gam = np.ascontiguousarray(gammas, dtype=np.int32)
    tok = None if draft_tokens is None else np.ascontiguousarray(draft_tokens, dtype=np.int32)
    B = len(gam)
    R_t = (int(offs[-1]) if B else 0) + B
    out_t = np.full((nsteps, R_t), -7, dtype=np.int32)
    out_n = np.full((nsteps, B), -7, dtype=np.int32)
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    st = lib().oracle_verify_steps(_ptr(target), _ptr(draft), dtype, _ptr(tok), _ptr(offs), _ptr(gam), B, V,
                                   float(temperature), seed, step0, int(nsteps), _ptr(out_t), _ptr(out_n),
                                   int(nthreads))
    return out_t, out_n, int(st)


def draw_bracket(trow, drow, V, temperature, u, k_query, x_excl=-1):
    """(token, C_{k-1}/S, C_k/S, S) of one inverse-CDF draw; see ``oracle_draw_bracket``
    (x_excl >= 0 with drow None: the residual of a point-mass draft at x_excl)."""
    trow = np.ascontiguousarray(trow)
    dtype = BF16 if trow.dtype == np.uint16 else F32
    if dtype == F32:
        trow = trow.astype(np.float32, copy=False)
    if drow is not None:
        drow = np.ascontiguousarray(drow).astype(trow.dtype, copy=False)
    lo = np.zeros(1); hi = np.zeros(1); S = np.zeros(1)
    tok = lib().oracle_draw_bracket(_ptr(trow), _ptr(drow), dtype, V, float(temperature), float(u),
                                    int(x_excl), int(k_query), _ptr(lo), _ptr(hi), _ptr(S))
    return tok, float(lo[0]), float(hi[0]), float(S[0])


def tree_probs(p, parents, x, u_acc, u_smp):
    """The tree rule on fp64 probabilities (see ``oracle_tree_probs``): p [gamma+1, V], parents/x of
    the gamma non-root nodes, u_acc/u_smp indexed by slot / node. Returns (n, tokens, path)."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    g = p.shape[0] - 1
    V = p.shape[1]
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(max(g, 1))
    xs = np.ascontiguousarray(x, dtype=np.int32).reshape(max(g, 1))
    ua = np.ascontiguousarray(u_acc, dtype=np.float64).reshape(max(g, 1))
    us = np.ascontiguousarray(u_smp, dtype=np.float64).reshape(g + 1)
    out = np.zeros(g + 1, dtype=np.int32)
    path = np.zeros(max(g, 1), dtype=np.int32)
    n = lib().oracle_tree_probs(_ptr(p), _ptr(par), _ptr(xs), g, V, _ptr(ua), _ptr(us), _ptr(out), _ptr(path))
    return n, out, path[:g]


def verify_tree(target, draft_tokens, seq_offsets, gammas, parents, V, temperature, seed, step):
    """Verify token trees (see ``oracle_verify_tree``). Returns (tokens, num_accepted, path, status)."""
    target = np.ascontiguousarray(target)
    dtype = BF16 if target.dtype == np.uint16 else F32
    if dtype == F32:
        target = target.astype(np.float32, copy=False)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    gam = np.ascontiguousarray(gammas, dtype=np.int32)
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    par = np.ascontiguousarray(parents, dtype=np.int32)
    B = len(gam)
    R_d = int(offs[-1]) if B else 0
    out = np.full(R_d + B, -7, dtype=np.int32)
    n = np.full(B, -7, dtype=np.int32)
    path = np.full(max(R_d, 1), -7, dtype=np.int32)
    st = lib().oracle_verify_tree(_ptr(target), dtype, _ptr(tok), _ptr(offs), _ptr(gam), _ptr(par), B, V,
                                  float(temperature), seed, step, _ptr(out), _ptr(n), _ptr(path))
    return out, n, path[:R_d], int(st)
