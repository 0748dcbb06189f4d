"""The optional parts of the encoder on the GPU against the oracle: the
embedding and final LayerNorms (the published ModernBERT layout), the
per-token (multi-vector) output with and without a projection, in every
arithmetic of the library, and the 4- and 6-bit weight-block integer paths
(W4A8, W6A8), through the C ABI.

Per-token vectors are held to the same bars as the pooled ones: fp32 max
|GPU - oracle| <= 1e-4; bf16 cosine >= 0.9995 and max abs <= 3e-3 per vector;
W8A8 (no outliers) cosine >= 0.9995 against the W8A8 oracle.
"""
import ctypes

import numpy as np
import pytest

import oracle
from text_embedding_encoder_gb300 import binding, synth

torch = pytest.importorskip("torch")
from gpu_util import BF16_COS, assert_embeddings_close, dev, make_encoder  # noqa: E402

pytestmark = pytest.mark.gpu

EXT = synth.Shape(**{**synth.TINY.as_dict(), "emb_norm": True, "final_norm": True, "proj_dim": 128})
NORMS_ONLY = synth.Shape(**{**synth.TINY.as_dict(), "emb_norm": True, "final_norm": True})
LENGTHS = [1, 2, 8, 37, 64, 65, 150, 129]


def _cos_rows(a, b):
    return np.sum(a * b, axis=1) / (np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1))


@pytest.mark.parametrize("shape", [EXT, NORMS_ONLY], ids=["norms+proj128", "norms"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_pooled_and_token_outputs(lib, shape, dtype):
    w = synth.make_weights(shape, seed=3, std=0.05)
    ids, cu = synth.make_batch(LENGTHS, shape.vocab, seed=4)
    enc = make_encoder(shape, dtype, w, max_tokens=1024, max_texts=16)
    model = oracle.OracleModel(w, shape, dtype)
    assert_embeddings_close(enc.encode(ids, cu), oracle.encode_packed(ids, cu, model), dtype)
    toks = enc.encode_tokens(ids, cu)
    assert toks.shape == (len(ids), shape.proj_dim or shape.hidden)
    want = oracle.encode_packed_tokens(ids, cu, model)
    assert_embeddings_close(toks, want, dtype)
    np.testing.assert_allclose(np.linalg.norm(toks, axis=1), 1.0, atol=1e-5)
    # the device path writes the same vectors
    d_out = torch.empty(len(ids), enc.token_width, device="cuda")
    enc.encode_tokens_device(dev(ids), dev(cu), cu, d_out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d_out.cpu().numpy(), toks)
    enc.close()


def test_token_output_w8a8(lib):
    shape = EXT
    w = synth.make_weights(shape, seed=5)
    ids, cu = synth.make_batch([8, 37, 64, 150], shape.vocab, seed=6)
    enc = make_encoder(shape, "w8a8", w, max_tokens=512, max_texts=8)
    toks = enc.encode_tokens(ids, cu)
    want = oracle.encode_packed_tokens(ids, cu, oracle.OracleModel(w, shape, "w8a8"))
    cos = _cos_rows(toks.astype(np.float64), want)
    assert cos.min() >= BF16_COS, cos.min()
    enc.close()


def test_ruri_token_output_bf16(lib):
    shape = synth.Shape(**{**synth.RURI_310M.as_dict(), "emb_norm": True, "final_norm": True, "proj_dim": 128})
    w = synth.make_weights(shape, seed=0)
    ids, cu = synth.make_batch([8, 57, 190], shape.vocab, seed=0)
    enc = make_encoder(shape, "bf16", w, max_tokens=512, max_texts=8)
    model = oracle.OracleModel(w, shape, "bf16")
    assert_embeddings_close(enc.encode_tokens(ids, cu), oracle.encode_packed_tokens(ids, cu, model), "bf16")
    assert_embeddings_close(enc.encode(ids, cu), oracle.encode_packed(ids, cu, model), "bf16")
    enc.close()


def test_optional_weights_and_output_are_validated(lib):
    shape = EXT
    w = synth.make_weights(shape, seed=3)
    enc = binding.Encoder(shape, "bf16", max_tokens=256, max_texts=8)
    w_missing = synth.make_weights(shape, seed=3)
    w_missing.w_proj = None
    with pytest.raises(binding.TeeError) as e:
        enc.load_weights(w_missing)
    assert e.value.code == binding.TEE_EINVAL
    enc.load_weights(w)
    ids, cu = synth.make_batch([5, 9], shape.vocab, seed=1)
    buf = torch.empty(len(ids) * 128 + 4, device="cuda")
    rc = enc.lib.tee_encode_tokens_device(enc.ctx, dev(ids).data_ptr(), dev(cu).data_ptr(),
                                          np.ascontiguousarray(cu).ctypes.data, 2, buf.data_ptr() + 4, None)
    assert rc == binding.TEE_EINVAL
    toks = enc.encode_tokens(ids, cu)   # the context is still usable
    assert np.all(np.isfinite(toks))
    assert enc.device_status() == 0
    enc.close()


# ---------------------------------------------------------------------------
# the 4- and 6-bit weight-block integer paths
# ---------------------------------------------------------------------------

ODD = synth.Shape(n_layers=2, hidden=384, n_heads=6, head_dim=64, intermediate=640, vocab=1000)


QUANT = {"w4a8": oracle.quantize_weight_blocks4, "w6a8": oracle.quantize_weight_blocks6}


@pytest.mark.parametrize("variant", ["w4a8", "w6a8"])
@pytest.mark.parametrize("which,name", [(0, "wqkv"), (1, "wo"), (2, "wi"), (3, "wo_ffn")])
def test_packed_weight_codes_and_block_sums_bit_exact(lib, variant, which, name):
    """4- and 6-bit weight blocks: the codes the library packed at load, read
    back and widened, and the scales equal the oracle's quantiser; the exact
    int32 block sums of the packed codes equal the oracle's integer sums."""
    shape = ODD
    w = synth.make_weights(shape, seed=21, outliers=True)
    enc = make_encoder(shape, variant, w, max_tokens=256, max_texts=8)
    layer = 1
    Wf = getattr(w, name)[layer]
    N, K = Wf.shape
    q_ref, d_ref = QUANT[variant](Wf)
    q_gpu = np.empty((N, K), np.int8)
    d_gpu = np.empty((N, K // 32), np.float32)
    enc.check(enc.lib.tee_weight_codes(enc.ctx, layer, which, q_gpu.ctypes.data, d_gpu.ctypes.data))
    np.testing.assert_array_equal(q_gpu, q_ref)
    np.testing.assert_array_equal(d_gpu.view(np.uint32), d_ref.view(np.uint32))
    rng = np.random.default_rng(8 + which)
    M = 141
    qa, _ = oracle.quantize_rows7((rng.standard_normal((M, K)) * 3).astype(np.float32))
    qa[0, :] = 63
    parts = torch.empty(M, N, K // 32, dtype=torch.int32, device="cuda")
    enc.op("tee_op_w8a8_partials", layer, which, dev(qa), M, parts, 0)
    np.testing.assert_array_equal(parts.cpu().numpy().astype(np.int64), oracle.int_block_partials(qa, q_ref))
    enc.close()


@pytest.mark.parametrize("variant", ["w4a8", "w6a8"])
def test_packed_weight_encode_tiny_and_ruri(lib, variant):
    for shape, lengths in ((synth.TINY, synth.TINY_LENGTHS), (synth.RURI_310M, synth.ACCURACY_LENGTHS)):
        w = synth.make_weights(shape, seed=0)
        ids, cu = synth.make_batch(lengths, shape.vocab, seed=0)
        enc = make_encoder(shape, variant, w, max_tokens=2048, max_texts=16)
        got = enc.encode(ids, cu).astype(np.float64)
        want = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, variant))
        cos = _cos_rows(got, want)
        ref32 = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "fp32"))
        print(f"{shape.n_layers}-layer {variant}: min cos vs {variant} oracle {cos.min():.6f}; "
              f"{variant} oracle vs fp32 oracle {_cos_rows(want, ref32).min():.4f}")
        assert cos.min() >= BF16_COS, cos.min()
        assert enc.device_status() == 0
        enc.close()


# ---------------------------------------------------------------------------
# weights from a checkpoint file, and the host front end around the encoder
# ---------------------------------------------------------------------------

def test_checkpoint_file_gives_identical_embeddings(lib, tmp_path):
    """Weights written to a safetensors file and read back load into the
    library bit-identically, so the embeddings are identical (F32 file); a
    BF16 file gives the embeddings of the bf16-rounded weights."""
    from text_embedding_encoder_gb300 import weights_io
    shape = synth.Shape(**{**synth.TINY.as_dict(), "emb_norm": True, "final_norm": True})
    w = synth.make_weights(shape, seed=8)
    ids, cu = synth.make_batch([37, 150, 8, 64], shape.vocab, seed=8)
    p = tmp_path / "ckpt.safetensors"
    weights_io.save_weights_file(p, w, shape, "F32")
    for dtype in ("fp32", "bf16"):
        a = make_encoder(shape, dtype, w, max_tokens=512, max_texts=8)
        b = make_encoder(shape, dtype, weights_io.load_weights_file(p, shape), max_tokens=512, max_texts=8)
        np.testing.assert_array_equal(a.encode(ids, cu), b.encode(ids, cu))
        a.close()
        b.close()
    weights_io.save_weights_file(p, w, shape, "BF16")
    enc = make_encoder(shape, "fp32", weights_io.load_weights_file(p, shape), max_tokens=512, max_texts=8)
    w16 = weights_io.load_weights_file(p, shape)
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(w16, shape, "fp32"))
    assert_embeddings_close(enc.encode(ids, cu), ref, "fp32")
    enc.close()


def test_front_end_segment_encode_similarity(lib):
    """Texts segmented by the Unigram front end, packed, encoded, and turned
    into the similarity matrix: unit diagonal, symmetric, equal to the dot
    products of the oracle's vectors of the same ids."""
    rng = np.random.default_rng(12)
    shape = synth.TINY
    alphabet = list("川べりでサーフボードを持った人たちがいます瑠璃色はどんな")
    pieces = ["<unk>", "<s>", "</s>"] + sorted(set(alphabet) | {"".join(rng.choice(alphabet, 2)) for _ in range(300)})
    pieces = pieces[:shape.vocab]
    scores = np.concatenate([[0, 0, 0], -rng.uniform(1, 9, len(pieces) - 3)]).astype(np.float32)
    tok = binding.Unigram(pieces, scores, 0, -20.0, synth.BOS_ID, synth.EOS_ID)
    texts = ["川べりでサーフボードを持った人たちがいます", "サーフボードを持った人たち", "瑠璃色はどんな色？", "色"]
    id_lists = [tok.encode(t) for t in texts]
    ids, cu = binding.pack_texts(id_lists)
    w = synth.make_weights(shape, seed=0)
    enc = make_encoder(shape, "bf16", w, max_tokens=512, max_texts=8)
    vecs = enc.encode(ids, cu)
    enc.close()
    sim = binding.similarity(vecs)
    np.testing.assert_allclose(np.diag(sim), 1.0, atol=2e-6)
    np.testing.assert_array_equal(sim, sim.T)
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "bf16"))
    np.testing.assert_allclose(sim, ref @ ref.T, atol=2e-3)
    print(binding.format_similarity(sim))
    tok.close()
