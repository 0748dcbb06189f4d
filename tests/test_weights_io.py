"""The safetensors weight importer (text_embedding_encoder_gb300.weights_io) on
the CPU: round trips through files written by the module's own writer (and by
its command line), exact widening of the stored dtypes, and refusals that name
the offending tensor."""
import json
import os
import struct
import subprocess
import sys

import numpy as np
import pytest

import oracle
from text_embedding_encoder_gb300 import synth, weights_io

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPE = synth.Shape(n_layers=3, hidden=256, n_heads=4, head_dim=64, intermediate=512, vocab=4096, emb_norm=True,
                    final_norm=True)


def _same(a, b):
    np.testing.assert_array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def _all_equal(w1, w2, conv=lambda a: a):
    _same(w1.tok_emb, conv(w2.tok_emb))
    for key in weights_io.PER_LAYER:
        for a, b in zip(getattr(w1, key), getattr(w2, key)):
            _same(a, conv(b))
    _same(w1.ln_emb, conv(w2.ln_emb))
    _same(w1.ln_final, conv(w2.ln_final))


def test_f32_round_trip_is_bit_identical(tmp_path):
    w = synth.make_weights(SHAPE, seed=5)
    p = tmp_path / "w.safetensors"
    weights_io.save_weights_file(p, w, SHAPE, "F32")
    _all_equal(weights_io.load_weights_file(p, SHAPE), w)
    # header: 8-byte length, JSON padded to 8 bytes, contiguous data ranges
    raw = p.read_bytes()
    (n,) = struct.unpack("<Q", raw[:8])
    assert n % 8 == 0
    header = json.loads(raw[8:8 + n])
    assert header["layers.2.mlp.Wi.weight"]["shape"] == [1024, 256]
    assert len(raw) == 8 + n + max(v["data_offsets"][1] for k, v in header.items() if k != "__metadata__")


def test_bf16_file_holds_the_bf16_rounded_weights(tmp_path):
    w = synth.make_weights(SHAPE, seed=6)
    p = tmp_path / "w16.safetensors"
    weights_io.save_weights_file(p, w, SHAPE, "BF16")
    _all_equal(weights_io.load_weights_file(p, SHAPE), w, conv=oracle.round_to_bf16)


def test_prefix_f16_and_refusals(tmp_path):
    w = synth.make_weights(SHAPE, seed=7)
    t = weights_io.tensors_from_weights(w, SHAPE)
    pref = {"model." + k: v for k, v in t.items()}
    p = tmp_path / "pref.safetensors"
    weights_io.write_safetensors(p, pref)
    _all_equal(weights_io.load_weights_file(p, SHAPE), w)
    # F16 storage widens exactly
    h = np.array([0.5, -2.0, 65504.0, 6.1e-5], np.float16)
    body = h.astype("<f2").tobytes()
    hdr = json.dumps({"x": {"dtype": "F16", "shape": [4], "data_offsets": [0, len(body)]}}).encode()
    hdr += b" " * (-len(hdr) % 8)
    q = tmp_path / "f16.safetensors"
    q.write_bytes(struct.pack("<Q", len(hdr)) + hdr + body)
    _same(weights_io.read_safetensors(q)["x"], h.astype(np.float32))
    # a missing tensor and a misshapen one are named
    del t["layers.1.mlp_norm.weight"]
    with pytest.raises(KeyError, match="layers.1.mlp_norm.weight"):
        weights_io.weights_from_tensors(t, SHAPE)
    t["layers.1.mlp_norm.weight"] = np.zeros(255, np.float32)
    with pytest.raises(ValueError, match="layers.1.mlp_norm.weight"):
        weights_io.weights_from_tensors(t, SHAPE)
    # a header length past the end of the file
    bad = tmp_path / "bad.safetensors"
    bad.write_bytes(struct.pack("<Q", 1 << 40) + b"{}")
    with pytest.raises(ValueError):
        weights_io.read_safetensors(bad)


def test_command_line_writes_a_loadable_checkpoint(tmp_path):
    p = tmp_path / "cli.safetensors"
    r = subprocess.run([sys.executable, "-m", "text_embedding_encoder_gb300.weights_io", str(p), "tiny", "F32", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    w = weights_io.load_weights_file(p, synth.TINY)
    _same(w.wqkv[1], synth.make_weights(synth.TINY, seed=3).wqkv[1])
