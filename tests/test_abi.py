"""The C ABI library builds, loads and exports every entry point include/dspark.h
declares; the Python structs match the C layout; host-side argument checks
return their status codes without touching a GPU (no GPU)."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

import mla_block_diffusion_gb300 as M
from mla_block_diffusion_gb300 import build as B
from synthetic.configs import FULL, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return M.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert set(names) == set(M.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (dspark_[a-z_]+)", out))
    assert set(names) <= exported
    for n in names:
        assert hasattr(L, n)


def test_struct_layout_matches_header(L):
    probe = r"""
#include <stdio.h>
#include <stddef.h>
#include "dspark.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(dspark_geom_t), sizeof(dspark_mat_t), sizeof(dspark_layer_weights_t),
         sizeof(dspark_weights_t), sizeof(dspark_kv_t), sizeof(dspark_sample_t));
  printf("%zu %zu %zu %zu %zu %zu\n", offsetof(dspark_geom_t, weight_format), offsetof(dspark_weights_t, final_norm),
         offsetof(dspark_weights_t, b_conf), offsetof(dspark_kv_t, max_ctx), offsetof(dspark_sample_t, seed),
         offsetof(dspark_layer_weights_t, w_down));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "p.c"), os.path.join(d, "p")
        open(src, "w").write(probe)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), src, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    sizes = [int(x) for x in lines[0].split()]
    offs = [int(x) for x in lines[1].split()]
    assert sizes == [C.sizeof(M.Geom), C.sizeof(M.dspark.Mat), C.sizeof(M.dspark.LayerWeights),
                     C.sizeof(M.dspark.Weights), C.sizeof(M.KV), C.sizeof(M.Sample)]
    assert offs == [M.Geom.weight_format.offset, M.dspark.Weights.final_norm.offset, M.dspark.Weights.b_conf.offset,
                    M.KV.max_ctx.offset, M.Sample.seed.offset, M.dspark.LayerWeights.w_down.offset]


def test_status_strings(L):
    for code in (0, 1, 2, 3, 4, 5, 6, 16, 17, 18):
        assert L.dspark_status_str(code).decode() != "unknown status"
    assert L.dspark_status_str(99).decode() == "unknown status"


def _fake_weights(G, align=256):
    """Weight struct whose pointers are non-null and aligned but never dereferenced."""
    w = M.dspark.Weights()
    p = lambda k: C.c_void_p(0x10000 + k * align)
    w.w_fc = M.dspark.Mat(p(1), None, 1.0)
    for l in range(G.n_layers):
        lw = w.layers[l]
        for j, f in enumerate(("attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_kv_b", "mlp_norm")):
            setattr(lw, f, p(10 + 20 * l + j))
        for j, f in enumerate(("w_q_b", "w_o", "w_gate", "w_up", "w_down")):
            setattr(lw, f, M.dspark.Mat(p(30 + 20 * l + j), None, 1.0))
    w.final_norm, w.w_lm, w.markov_w1, w.markov_w2, w.w_conf = p(2), p(3), p(4), p(5), p(6)
    return w


def test_host_argument_checks(L):
    h = C.c_void_p()
    g = M.geom_struct(TINY)
    w = _fake_weights(TINY)
    assert L.dspark_create(None, C.byref(w), C.byref(h)) == 1
    bad = M.geom_struct(TINY)
    bad.hidden = 0
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 3
    bad = M.geom_struct(TINY)
    bad.hidden = 520  # not a multiple of 64
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 4
    bad = M.geom_struct(TINY)
    bad.kv_lora, bad.d_rope = 128, 48  # no attention kernel for (176, 128)
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 4
    bad = M.geom_struct(FULL)
    bad.vocab = 1 << 18
    assert L.dspark_create(C.byref(bad), C.byref(_fake_weights(FULL)), C.byref(h)) == 4
    bad = M.geom_struct(TINY, weight_format=7)  # no such format
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 4
    bad = M.geom_struct(TINY, weight_format=M.FMT_FP8)  # FP8 needs per-channel scales
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 1
    bad = M.geom_struct(TINY, weight_format=M.FMT_NVFP4)  # q_lora 128: group-scale rows not 16-byte strides
    assert L.dspark_create(C.byref(bad), C.byref(w), C.byref(h)) == 4
    w2 = _fake_weights(TINY)
    w2.layers[1].w_up = M.dspark.Mat(None, None, 1.0)
    assert L.dspark_create(C.byref(g), C.byref(w2), C.byref(h)) == 1
    w3 = _fake_weights(TINY)
    w3.w_lm = C.c_void_p(0x10008)
    assert L.dspark_create(C.byref(g), C.byref(w3), C.byref(h)) == 2
    # calls on a null handle fail fast
    assert L.dspark_workspace_bytes(None, 1, 128) == 0
    s = M.Sample(0, 0, 1.0, 1.0, 0, 0)
    assert L.dspark_fuse_ctx(None, None, None, 1, None, 0, None) == 1
    assert L.dspark_draft_block(None, None, None, None, None, 1, None, 0, None) == 1
    assert L.dspark_markov_rollout(None, None, None, C.byref(s), None, None, 1, None, 0, None) == 1
    assert L.dspark_confidence(None, None, None, 1, None) == 1
    assert L.dspark_verify(None, None, None, None, C.byref(s), None, None, 1, None, 0, None) == 1
    assert L.dspark_check(None, None, None) == 1
