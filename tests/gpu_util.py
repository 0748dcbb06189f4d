"""Shared helpers of the GPU tests: device buffers and tolerances.

The tolerances are those the encoder is held to:
  fp32 path  max |GPU - oracle| <= 1e-4 per element of the final embeddings;
  bf16 path  cosine >= 0.9995 and max |GPU - oracle| <= 3e-3 per embedding;
  integer path: int8 codes and int32 block sums bit-exact.
For single steps on bf16 activations the GPU rounds its output to bf16
(relative error 2^-9), so step checks use a relative bound on top of that.
"""
import numpy as np
import torch

from text_embedding_encoder_gb300 import binding
import oracle

FP32_ABS = 1e-4
BF16_COS = 0.9995
BF16_ABS = 3e-3


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def act_dtype(dt):
    return torch.bfloat16 if dt == "bf16" else torch.float32


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def make_encoder(shape, dtype, weights, max_tokens, max_texts=4096):
    enc = binding.Encoder(shape, dtype, max_tokens=max_tokens, max_texts=max_texts)
    enc.load_weights(weights)
    return enc


def assert_step_close(got, ref, dtype, fp32_atol=2e-5, bf16_rel=1.2e-2):
    """Single-step check: fp32 within an absolute bound; bf16 within a bound
    relative to the output scale (one bf16 rounding of the output plus the
    rounding of bf16 inputs, which the oracle sees exactly)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    if dtype == "bf16":
        scale = np.abs(ref).max() + 1e-30
        assert err.max() <= bf16_rel * scale, (err.max(), scale)
        rel_fro = np.linalg.norm(got - ref) / (np.linalg.norm(ref) + 1e-30)
        assert rel_fro <= 4e-3, rel_fro
    else:
        assert err.max() <= fp32_atol * max(1.0, np.abs(ref).max()), err.max()


def assert_embeddings_close(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    if dtype == "fp32":
        assert err <= FP32_ABS, err
    else:
        cos = np.sum(got * ref, axis=1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1))
        assert cos.min() >= BF16_COS, cos.min()
        assert err <= BF16_ABS, err
    return err
