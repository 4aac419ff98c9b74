"""ORACLE (test infrastructure only): ctypes access to the oracle's C sampling,
Markov rollout and verification routines in ``sampling.c``.

Only tests, the smoke check and the benchmark's CPU-baseline leg use this.
"""
from __future__ import annotations

import ctypes as C
from typing import Tuple

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        L = _lib
        u32p = C.POINTER(C.c_uint32)
        L.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.oracle_uniform_u32.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
        L.oracle_uniform_u32.restype = C.c_uint32
        L.oracle_exp_hat.argtypes = [C.c_float]
        L.oracle_exp_hat.restype = C.c_float
        L.oracle_top_p_q32.argtypes = [C.c_float]
        L.oracle_top_p_q32.restype = C.c_uint64
        L.oracle_row_weights.argtypes = [C.c_void_p, C.c_int, C.c_float, C.c_void_p]
        L.oracle_nucleus.argtypes = [C.c_void_p, C.c_int, C.c_float, C.c_void_p]
        L.oracle_sample_nucleus.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_uint64, C.c_uint32]
        L.oracle_sample_nucleus.restype = C.c_int32
        L.oracle_argmax.argtypes = [C.c_void_p, C.c_int, C.c_void_p]
        L.oracle_markov_rollout.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                            C.c_int32, C.c_int, C.c_float, C.c_float, C.c_uint64,
                                            C.c_uint32, C.c_uint32, C.c_void_p, C.c_void_p]
        L.oracle_verify_greedy.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_verify_prob_core.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                              C.c_float, C.c_float, C.c_void_p, C.c_void_p, C.c_uint32,
                                              C.c_void_p, C.c_void_p]
        L.oracle_verify_prob.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                         C.c_float, C.c_float, C.c_uint64, C.c_uint32, C.c_uint32,
                                         C.c_void_p, C.c_void_p]
        vp = C.c_void_p
        L.oracle_verify_block_stats.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp]
        L.oracle_block_residual_weights.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float,
                                                    C.c_int, C.c_double, vp]
        L.oracle_verify_block_core.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp,
                                               C.c_uint32, vp, vp]
        L.oracle_verify_block.argtypes = [vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, C.c_uint64,
                                          C.c_uint32, C.c_uint32, vp, vp]
    return _lib


class OracleError(RuntimeError):
    pass


def _chk(st: int):
    if st != 0:
        raise OracleError(f"oracle status {st}")


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


class Nucleus(C.Structure):
    _fields_ = [("S", C.c_uint64), ("kstar", C.c_uint64), ("Sn", C.c_uint64), ("size", C.c_int32)]


def philox4x32_10(ctr, key) -> Tuple[int, int, int, int]:
    c = (C.c_uint32 * 4)(*ctr)
    k = (C.c_uint32 * 2)(*key)
    o = (C.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, o)
    return tuple(o)


def uniform_u32(seed: int, seq: int, step: int, pos: int, purpose: int) -> int:
    return lib().oracle_uniform_u32(seed, seq, step, pos, purpose)


def exp_hat(x: float) -> float:
    return lib().oracle_exp_hat(x)


def top_p_q32(top_p: float) -> int:
    return lib().oracle_top_p_q32(top_p)


def row_weights(l: np.ndarray, T: float) -> np.ndarray:
    l = np.ascontiguousarray(l, dtype=np.float32)
    E = np.zeros(l.shape[0], dtype=np.uint64)
    _chk(lib().oracle_row_weights(_ptr(l), l.shape[0], T, _ptr(E)))
    return E


def nucleus(E: np.ndarray, top_p: float) -> Nucleus:
    E = np.ascontiguousarray(E, dtype=np.uint64)
    n = Nucleus()
    _chk(lib().oracle_nucleus(_ptr(E), E.shape[0], top_p, C.byref(n)))
    return n


def sample_nucleus(E: np.ndarray, kstar: int, Sn: int, W24: int) -> int:
    E = np.ascontiguousarray(E, dtype=np.uint64)
    return lib().oracle_sample_nucleus(_ptr(E), E.shape[0], kstar, Sn, W24)


def argmax(l: np.ndarray) -> int:
    l = np.ascontiguousarray(l, dtype=np.float32)
    o = C.c_int32()
    _chk(lib().oracle_argmax(_ptr(l), l.shape[0], C.byref(o)))
    return o.value


def _u16(a) -> np.ndarray:
    """bf16 bytes as uint16 (accepts a torch bf16 tensor or a uint16 array)."""
    if hasattr(a, "view") and hasattr(a, "cpu"):
        import torch
        return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(a, dtype=np.uint16)


def markov_rollout(z: np.ndarray, w1_bf16, w2_bf16, anchor: int, draft_mode: int = 0, T: float = 1.0,
                   top_p: float = 1.0, seed: int = 0, seq: int = 0, step: int = 0):
    """One sequence: z fp32 [B, V]; w1 bf16 [V, r]; w2 bf16 [r, V] -> (tokens [B], ell [B, V])."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    B, V = z.shape
    w1 = _u16(w1_bf16)
    w2 = _u16(w2_bf16)
    r = w1.shape[1]
    assert w1.shape == (V, r) and w2.shape == (r, V)
    tokens = np.zeros(B, dtype=np.int32)
    ell = np.zeros((B, V), dtype=np.float32)
    _chk(lib().oracle_markov_rollout(_ptr(z), B, V, r, _ptr(w1), _ptr(w2), int(anchor), draft_mode, T,
                                     top_p, seed, seq, step, _ptr(tokens), _ptr(ell)))
    return tokens, ell


def verify_greedy(P: np.ndarray, tokens: np.ndarray):
    P = np.ascontiguousarray(P, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B = tokens.shape[0]
    assert P.shape[0] == B + 1
    a = C.c_int32()
    out = np.zeros(B + 1, dtype=np.int32)
    _chk(lib().oracle_verify_greedy(_ptr(P), _ptr(tokens), B, P.shape[1], C.byref(a), _ptr(out)))
    return a.value, out


def verify_prob_core(P, ell, tokens, draft_greedy: int, T: float, top_p: float, U, Wres, Wbonus: int):
    P = np.ascontiguousarray(P, dtype=np.float32)
    ell = np.ascontiguousarray(ell, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B = tokens.shape[0]
    U = np.ascontiguousarray(U, dtype=np.uint32)
    Wres = np.ascontiguousarray(Wres, dtype=np.uint32)
    a = C.c_int32()
    out = np.zeros(B + 1, dtype=np.int32)
    _chk(lib().oracle_verify_prob_core(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T, top_p,
                                       _ptr(U), _ptr(Wres), Wbonus, C.byref(a), _ptr(out)))
    return a.value, out


def verify_prob(P, ell, tokens, draft_greedy: int, T: float, top_p: float, seed: int, seq: int, step: int):
    P = np.ascontiguousarray(P, dtype=np.float32)
    ell = np.ascontiguousarray(ell, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B = tokens.shape[0]
    a = C.c_int32()
    out = np.zeros(B + 1, dtype=np.int32)
    _chk(lib().oracle_verify_prob(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T, top_p,
                                  seed, seq, step, C.byref(a), _ptr(out)))
    return a.value, out


def _vargs(P, ell, tokens):
    P = np.ascontiguousarray(P, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B = tokens.shape[0]
    ell = np.ascontiguousarray(ell if ell is not None else np.zeros((max(B, 1), P.shape[1])), dtype=np.float32)
    return P, ell, tokens, B


def block_stats(P, ell, tokens, draft_greedy: int, T: float, top_p: float):
    """Block verification's pi_0..pi_B and h_0..h_B (h_0 = 0) for one drafted block."""
    P, ell, tokens, B = _vargs(P, ell, tokens)
    pi = np.zeros(B + 1)
    h = np.zeros(B + 1)
    _chk(lib().oracle_verify_block_stats(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T, top_p,
                                         _ptr(pi), _ptr(h)))
    return pi, h


def block_residual_weights(P, ell, tokens, draft_greedy: int, T: float, top_p: float, i: int, pi: float):
    """Fixed-point (2^-80) residual weights max(pi p_i - q_i, 0) of position i, as Python ints."""
    P, ell, tokens, B = _vargs(P, ell, tokens)
    w = np.zeros(2 * P.shape[1], dtype=np.uint64)
    _chk(lib().oracle_block_residual_weights(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T,
                                             top_p, i, pi, _ptr(w)))
    return [int(w[2 * v]) | (int(w[2 * v + 1]) << 64) for v in range(P.shape[1])]


def verify_block_core(P, ell, tokens, draft_greedy: int, T: float, top_p: float, U, Wres, Wbonus: int):
    P, ell, tokens, B = _vargs(P, ell, tokens)
    U = np.ascontiguousarray(U, dtype=np.uint32)
    Wres = np.ascontiguousarray(Wres, dtype=np.uint32)
    a = C.c_int32()
    out = np.zeros(B + 1, dtype=np.int32)
    _chk(lib().oracle_verify_block_core(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T, top_p,
                                        _ptr(U), _ptr(Wres), Wbonus, C.byref(a), _ptr(out)))
    return a.value, out


def verify_block(P, ell, tokens, draft_greedy: int, T: float, top_p: float, seed: int, seq: int, step: int):
    P, ell, tokens, B = _vargs(P, ell, tokens)
    a = C.c_int32()
    out = np.zeros(B + 1, dtype=np.int32)
    _chk(lib().oracle_verify_block(_ptr(P), _ptr(ell), _ptr(tokens), B, P.shape[1], draft_greedy, T, top_p, seed,
                                   seq, step, C.byref(a), _ptr(out)))
    return a.value, out
