"""Thin Python binding of libdspark (include/dspark.h) over ctypes.

Argument marshalling only: every step of the draft-and-verify path runs in the
library's CUDA kernels. torch provides device memory and the stream. There is
no fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdspark.so")

MAX_LAYERS = 16
GREEDY, PROBABILISTIC, BLOCK = 0, 1, 2
FMT_BF16, FMT_FP8, FMT_NVFP4, FMT_MXFP4 = 0, 1, 2, 3

STATUS = {0: "OK", 1: "ERR_NULL", 2: "ERR_ALIGN", 3: "ERR_SHAPE", 4: "ERR_UNSUPPORTED", 5: "ERR_CUDA",
          6: "ERR_WORKSPACE", 16: "ERR_TIMEOUT", 17: "ERR_BAD_INPUT", 18: "ERR_OOB"}
EXPORTS = ("dspark_create", "dspark_destroy", "dspark_workspace_bytes", "dspark_fuse_ctx", "dspark_draft_block",
           "dspark_markov_rollout", "dspark_confidence", "dspark_verify", "dspark_check", "dspark_status_str",
           "dspark_fuse_ctx_noalloc", "dspark_kv_append")


class Geom(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("hidden", "n_aux", "n_layers", "n_heads", "q_lora", "kv_lora", "d_nope",
                                       "d_rope", "d_v", "inter", "vocab", "rank", "block")] + [
        ("rope_theta", C.c_float), ("eps", C.c_float), ("yarn_factor", C.c_float), ("yarn_orig_ctx", C.c_int),
        ("yarn_alpha", C.c_float), ("yarn_beta", C.c_float), ("page_size", C.c_int), ("weight_format", C.c_int)]


class Mat(C.Structure):
    _fields_ = [("data", C.c_void_p), ("scale", C.c_void_p), ("global_scale", C.c_float)]


class LayerWeights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("w_qkv_a", C.c_void_p), ("q_a_norm", C.c_void_p),
                ("kv_a_norm", C.c_void_p), ("w_q_b", Mat), ("w_kv_b", C.c_void_p), ("w_o", Mat),
                ("mlp_norm", C.c_void_p), ("w_gate", Mat), ("w_up", Mat), ("w_down", Mat)]


class Weights(C.Structure):
    _fields_ = [("w_fc", Mat), ("layers", LayerWeights * MAX_LAYERS), ("final_norm", C.c_void_p),
                ("w_lm", C.c_void_p), ("markov_w1", C.c_void_p), ("markov_w2", C.c_void_p),
                ("w_conf", C.c_void_p), ("b_conf", C.c_float)]


class KV(C.Structure):
    _fields_ = [("pools", C.c_void_p * MAX_LAYERS), ("n_pages", C.c_int), ("page_table", C.c_void_p),
                ("max_pages", C.c_int), ("ctx_len", C.c_void_p), ("max_ctx", C.c_int)]


class Sample(C.Structure):
    _fields_ = [("draft_mode", C.c_int), ("verify_mode", C.c_int), ("temperature", C.c_float),
                ("top_p", C.c_float), ("seed", C.c_uint64), ("step", C.c_uint32)]


class DSparkError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({status})")
        self.status = status


_lib = None


def lib():
    """Load libdspark.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdspark.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        L.dspark_create.argtypes = [C.POINTER(Geom), C.POINTER(Weights), C.POINTER(vp)]
        L.dspark_destroy.argtypes = [vp]
        L.dspark_destroy.restype = None
        L.dspark_workspace_bytes.argtypes = [vp, i, i]
        L.dspark_workspace_bytes.restype = sz
        L.dspark_fuse_ctx.argtypes = [vp, vp, vp, i, vp, sz, vp]
        L.dspark_draft_block.argtypes = [vp, vp, C.POINTER(KV), vp, vp, i, vp, sz, vp]
        L.dspark_markov_rollout.argtypes = [vp, vp, vp, C.POINTER(Sample), vp, vp, i, vp, sz, vp]
        L.dspark_confidence.argtypes = [vp, vp, vp, i, vp]
        L.dspark_verify.argtypes = [vp, vp, vp, vp, C.POINTER(Sample), vp, vp, i, vp, sz, vp]
        L.dspark_check.argtypes = [vp, vp, vp]
        L.dspark_fuse_ctx_noalloc.argtypes = [vp, vp, vp, i, vp]
        L.dspark_kv_append.argtypes = [vp, vp, i, vp, C.POINTER(KV), i, vp, sz, vp]
        L.dspark_status_str.argtypes = [i]
        L.dspark_status_str.restype = C.c_char_p
        for f in EXPORTS:
            if f not in ("dspark_destroy", "dspark_workspace_bytes", "dspark_status_str"):
                getattr(L, f).restype = i
        _lib = L
    return _lib


def geom_struct(G, weight_format: int = FMT_BF16) -> Geom:
    return Geom(hidden=G.hidden, n_aux=G.n_aux, n_layers=G.n_layers, n_heads=G.n_heads, q_lora=G.q_lora,
                kv_lora=G.kv_lora, d_nope=G.d_nope, d_rope=G.d_rope, d_v=G.d_v, inter=G.inter, vocab=G.vocab,
                rank=G.rank, block=G.block, rope_theta=G.rope_theta, eps=G.eps, yarn_factor=G.yarn_factor,
                yarn_orig_ctx=G.yarn_orig_ctx, yarn_alpha=G.yarn_alpha, yarn_beta=G.yarn_beta,
                page_size=G.page_size, weight_format=weight_format)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _mat(v) -> "Mat":
    """A matrix entry: a bf16 tensor, or (data, scale, global_scale) for FP8 / NVFP4."""
    if isinstance(v, tuple):
        d, sc, g = v
        return Mat(_p(d), _p(sc), float(g))
    return Mat(_p(v), None, 1.0)


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _chk(fn: str, st: int):
    if st != 0:
        raise DSparkError(fn, st)


class DSpark:
    """One drafter (geometry + device-resident weights) bound to libdspark.

    ``W`` maps names to device tensors (bf16 matrices row-major [out, in], fp32
    norm gains and confidence head), as produced by the seeded generators. With
    ``weight_format`` FP8 or NVFP4 the quantised matrices (fc, q_b, o, gate, up,
    down) are (data, scale, global_scale) triples.
    The workspace is allocated here, zero-filled, for up to ``max_bs``
    sequences and contexts of ``max_ctx`` tokens.
    """

    def __init__(self, G, W: Dict[str, torch.Tensor], max_bs: int = 1, max_ctx: int = 0,
                 weight_format: int = FMT_BF16):
        self.G = G
        self.W = W
        L = lib()
        self.geom = geom_struct(G, weight_format)
        w = Weights()
        w.w_fc = _mat(W["w_fc"])
        for l in range(G.n_layers):
            P = f"l{l}."
            lw = w.layers[l]
            lw.attn_norm = _p(W[P + "attn_norm"])
            lw.w_qkv_a = _p(W[P + "w_qkv_a"])
            lw.q_a_norm = _p(W[P + "q_a_norm"])
            lw.kv_a_norm = _p(W[P + "kv_a_norm"])
            lw.w_q_b = _mat(W[P + "w_q_b"])
            lw.w_kv_b = _p(W[P + "w_kv_b"])
            lw.w_o = _mat(W[P + "w_o"])
            lw.mlp_norm = _p(W[P + "mlp_norm"])
            lw.w_gate = _mat(W[P + "w_gate"])
            lw.w_up = _mat(W[P + "w_up"])
            lw.w_down = _mat(W[P + "w_down"])
        w.final_norm = _p(W["final_norm"])
        w.w_lm = _p(W["w_lm"])
        w.markov_w1 = _p(W["markov_w1"])
        w.markov_w2 = _p(W["markov_w2"])
        w.w_conf = _p(W["w_conf"])
        w.b_conf = float(W["b_conf"].item()) if torch.is_tensor(W["b_conf"]) else float(W["b_conf"])
        self.weights = w
        h = C.c_void_p()
        _chk("dspark_create", L.dspark_create(C.byref(self.geom), C.byref(w), C.byref(h)))
        self.h = h
        self.max_bs, self.max_ctx = max_bs, max_ctx
        self.ws_bytes = L.dspark_workspace_bytes(h, max_bs, max_ctx)
        if self.ws_bytes == 0:
            raise DSparkError("dspark_workspace_bytes", 3)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device="cuda")

    def close(self):
        if getattr(self, "h", None):
            lib().dspark_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- the five calls ------------------------------------------------------------
    def fuse_ctx(self, aux: torch.Tensor, x: torch.Tensor, bs: int):
        _chk("dspark_fuse_ctx", lib().dspark_fuse_ctx(self.h, _p(aux), _p(x), bs, _p(self.ws), self.ws_bytes,
                                                       _stream()))

    def fuse_ctx_noalloc(self, aux: torch.Tensor, x: torch.Tensor, bs: int):
        """fc fusion with the library's own fixed scratch instead of the workspace."""
        _chk("dspark_fuse_ctx_noalloc", lib().dspark_fuse_ctx_noalloc(self.h, _p(aux), _p(x), bs, _stream()))

    def make_kv(self, pools: Sequence[torch.Tensor], page_table: torch.Tensor, ctx_len: torch.Tensor,
                max_ctx: int) -> KV:
        kv = KV()
        # the struct holds raw device pointers: keep the tensors alive as long as it lives
        kv._keep = (list(pools), page_table, ctx_len)
        for l, t in enumerate(pools):
            kv.pools[l] = t.data_ptr()
        kv.n_pages = int(pools[0].shape[0])
        kv.page_table = page_table.data_ptr()
        kv.max_pages = int(page_table.shape[1])
        kv.ctx_len = ctx_len.data_ptr()
        kv.max_ctx = int(max_ctx)
        return kv

    def draft_block(self, x: torch.Tensor, kv: KV, h_out: torch.Tensor, z: torch.Tensor, bs: int):
        _chk("dspark_draft_block", lib().dspark_draft_block(self.h, _p(x), C.byref(kv), _p(h_out), _p(z), bs,
                                                             _p(self.ws), self.ws_bytes, _stream()))

    def markov_rollout(self, z, anchor, sample: Sample, tokens, ell, bs: int):
        _chk("dspark_markov_rollout", lib().dspark_markov_rollout(self.h, _p(z), _p(anchor), C.byref(sample),
                                                                   _p(tokens), _p(ell), bs, _p(self.ws),
                                                                   self.ws_bytes, _stream()))

    def confidence(self, h_out, conf, bs: int):
        _chk("dspark_confidence", lib().dspark_confidence(self.h, _p(h_out), _p(conf), bs, _stream()))

    def verify(self, target_logits, ell, tokens, sample: Sample, accept_len, out_tokens, bs: int):
        _chk("dspark_verify", lib().dspark_verify(self.h, _p(target_logits), _p(ell), _p(tokens), C.byref(sample),
                                                   _p(accept_len), _p(out_tokens), bs, _p(self.ws), self.ws_bytes,
                                                   _stream()))

    def kv_append(self, x_new: torch.Tensor, n_new: torch.Tensor, kv: KV, bs: int):
        """Write the latent entries of newly verified tokens (x_new [bs, n_max, H]) into every
        layer's page pool at ctx_len + j, then advance ctx_len by n_new (device, in place)."""
        n_max = int(x_new.shape[1])
        _chk("dspark_kv_append", lib().dspark_kv_append(self.h, _p(x_new), n_max, _p(n_new), C.byref(kv), bs,
                                                         _p(self.ws), self.ws_bytes, _stream()))

    def check(self) -> int:
        """Synchronise and return (and clear) the device error word."""
        return lib().dspark_check(self.h, _p(self.ws), _stream())

    def check_noalloc(self) -> int:
        """Synchronise and return (and clear) the error word of the allocation-free fusion's fixed scratch."""
        return lib().dspark_check(self.h, None, _stream())
