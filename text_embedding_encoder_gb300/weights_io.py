"""Encoder weights to and from safetensors files.

The tensai page "テキスト埋め込み" (introduction) checks its encoder against the
trained Ruri v3 310m weights -- a ModernBERT checkpoint -- and matches the
model card's similarity matrix to within 0.003.  Trained weights are loaded
through this module: a safetensors file (an 8-byte little-endian header
length, a JSON header naming each tensor's dtype, shape and byte range, then
the raw little-endian data) is read into the fp32 host layout that
``Encoder.load_weights`` / ``tee_load_weights`` take.

Tensor names default to the published ModernBERT checkpoint layout as this
project reads it (an optional ``model.`` prefix is accepted):

  embeddings.tok_embeddings.weight   [V, H]     tok_emb
  embeddings.norm.weight             [H]        ln_emb    (Shape.emb_norm)
  layers.{l}.attn_norm.weight        [H]        ln_attn[l]
  layers.{l}.attn.Wqkv.weight        [3H, H]    wqkv[l]   rows q, k, v
  layers.{l}.attn.Wo.weight          [H, H]     wo[l]
  layers.{l}.mlp_norm.weight         [H]        ln_mlp[l]
  layers.{l}.mlp.Wi.weight           [2I, H]    wi[l]     rows: GELU input, then gate
  layers.{l}.mlp.Wo.weight           [H, I]     wo_ffn[l]
  final_norm.weight                  [H]        ln_final  (Shape.final_norm)

Every tensor the shape needs must be present with exactly that shape; a
missing or misshapen one is an error that names it.  (The page's encoder has
a LayerNorm in front of the attention of every layer; a checkpoint without
one for some layer cannot be represented and is refused.)  Stored dtypes F32,
F16 and BF16 are widened to fp32 exactly.  Host-side only: nothing here
touches a GPU.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np

from .synth import Weights

_NP = {"F32": np.dtype("<f4"), "F16": np.dtype("<f2"), "BF16": np.dtype("<u2")}

MODERNBERT_NAMES = {
    "tok_emb": "embeddings.tok_embeddings.weight",
    "ln_emb": "embeddings.norm.weight",
    "ln_attn": "layers.{l}.attn_norm.weight",
    "wqkv": "layers.{l}.attn.Wqkv.weight",
    "wo": "layers.{l}.attn.Wo.weight",
    "ln_mlp": "layers.{l}.mlp_norm.weight",
    "wi": "layers.{l}.mlp.Wi.weight",
    "wo_ffn": "layers.{l}.mlp.Wo.weight",
    "ln_final": "final_norm.weight",
}
PER_LAYER = ("ln_attn", "wqkv", "wo", "ln_mlp", "wi", "wo_ffn")


def _bf16_bits(a) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _widen(raw: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "BF16":
        return (raw.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return raw.astype(np.float32)


def read_safetensors(path) -> dict:
    """All tensors of a safetensors file as fp32 numpy arrays, by name."""
    size = os.path.getsize(path)
    with open(path, "rb") as f:
        head = f.read(8)
        if len(head) != 8:
            raise ValueError(f"{path}: not a safetensors file (shorter than its header length)")
        (n,) = struct.unpack("<Q", head)
        if n > size - 8:
            raise ValueError(f"{path}: header length {n} exceeds the file")
        header = json.loads(f.read(n).decode("utf-8"))
        base = 8 + n
        out = {}
        for name, info in header.items():
            if name == "__metadata__":
                continue
            dt = info["dtype"]
            if dt not in _NP:
                raise ValueError(f"{path}: tensor {name} has dtype {dt}; only F32, F16 and BF16 are read")
            shape = tuple(int(x) for x in info["shape"])
            b0, b1 = (int(x) for x in info["data_offsets"])
            count = int(np.prod(shape)) if shape else 1
            if b1 - b0 != count * _NP[dt].itemsize or base + b1 > size or b0 < 0:
                raise ValueError(f"{path}: tensor {name}: byte range [{b0}, {b1}) does not fit shape {shape}")
            f.seek(base + b0)
            raw = np.frombuffer(f.read(b1 - b0), dtype=_NP[dt]).reshape(shape)
            out[name] = _widen(raw, dt)
    return out


def write_safetensors(path, tensors: dict, dtype: str = "F32", metadata: dict | None = None) -> None:
    """Write fp32 arrays as one safetensors file, stored as F32 or BF16 (rounded
    to nearest even).  The header is padded with spaces to a multiple of 8 bytes."""
    if dtype not in ("F32", "BF16"):
        raise ValueError("dtype must be F32 or BF16")
    header, blobs, off = {}, [], 0
    for name in sorted(tensors):
        a = np.ascontiguousarray(tensors[name], dtype=np.float32)
        raw = a.astype("<f4").tobytes() if dtype == "F32" else _bf16_bits(a).astype("<u2").tobytes()
        header[name] = {"dtype": dtype, "shape": list(a.shape), "data_offsets": [off, off + len(raw)]}
        blobs.append(raw)
        off += len(raw)
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    hb = json.dumps(header, separators=(",", ":")).encode("utf-8")
    hb += b" " * (-len(hb) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(hb)))
        f.write(hb)
        for b in blobs:
            f.write(b)


def weights_from_tensors(tensors: dict, shape, names: dict = MODERNBERT_NAMES) -> Weights:
    """Map named fp32 tensors onto the encoder's weight layout for ``shape``."""
    H, I, V, L = shape.hidden, shape.intermediate, shape.vocab, shape.n_layers
    prefix = ""
    if names["tok_emb"] not in tensors and ("model." + names["tok_emb"]) in tensors:
        prefix = "model."

    def get(key, want, l=None):
        name = prefix + names[key].format(l=l)
        if name not in tensors:
            raise KeyError(f"tensor {name} ({key}) is missing")
        a = tensors[name]
        if tuple(a.shape) != want:
            raise ValueError(f"tensor {name} ({key}) has shape {tuple(a.shape)}, expected {want}")
        return np.ascontiguousarray(a, dtype=np.float32)

    want = {"ln_attn": (H,), "wqkv": (3 * H, H), "wo": (H, H), "ln_mlp": (H,), "wi": (2 * I, H), "wo_ffn": (H, I)}
    w = Weights(tok_emb=get("tok_emb", (V, H)))
    for l in range(L):
        for key in PER_LAYER:
            getattr(w, key).append(get(key, want[key], l))
    if getattr(shape, "emb_norm", False):
        w.ln_emb = get("ln_emb", (H,))
    if getattr(shape, "final_norm", False):
        w.ln_final = get("ln_final", (H,))
    return w


def tensors_from_weights(w: Weights, shape, names: dict = MODERNBERT_NAMES) -> dict:
    """The inverse of ``weights_from_tensors`` (no prefix)."""
    t = {names["tok_emb"]: w.tok_emb}
    for l in range(shape.n_layers):
        for key in PER_LAYER:
            t[names[key].format(l=l)] = getattr(w, key)[l]
    if getattr(shape, "emb_norm", False):
        t[names["ln_emb"]] = w.ln_emb
    if getattr(shape, "final_norm", False):
        t[names["ln_final"]] = w.ln_final
    return t


def load_weights_file(path, shape, names: dict = MODERNBERT_NAMES) -> Weights:
    """Read a safetensors checkpoint into the encoder's fp32 host layout."""
    return weights_from_tensors(read_safetensors(path), shape, names)


def save_weights_file(path, w: Weights, shape, dtype: str = "F32", names: dict = MODERNBERT_NAMES) -> None:
    """Write the encoder's weights as a safetensors checkpoint (F32 or BF16)."""
    write_safetensors(path, tensors_from_weights(w, shape, names), dtype,
                      metadata={"layout": "modernbert-style encoder", "hidden": shape.hidden,
                                "layers": shape.n_layers})


if __name__ == "__main__":
    # write the seeded synthetic weights of a shape as a checkpoint file:
    #   python -m text_embedding_encoder_gb300.weights_io OUT.safetensors [tiny|310m] [F32|BF16] [seed]
    import sys
    from . import synth
    out = sys.argv[1]
    shp = {"tiny": synth.TINY, "310m": synth.RURI_310M}[sys.argv[2] if len(sys.argv) > 2 else "tiny"]
    dt = sys.argv[3] if len(sys.argv) > 3 else "F32"
    seed = int(sys.argv[4]) if len(sys.argv) > 4 else 0
    save_weights_file(out, synth.make_weights(shp, seed=seed), shp, dt)
    print(out)
