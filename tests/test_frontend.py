"""The host-side front end (include/tee_frontend.h) on the CPU: the Unigram
max-score segmenter and the similarity matrix.

tensai page "テキスト埋め込み", §何が動くか (トークン化): the text is split into
the vocabulary pieces whose scores add up to the largest total and wrapped in
<s> ... </s>.  The segmenter is pinned by brute force: every way of cutting a
short text into pieces (or unknown single characters) is enumerated and
scored, and the library's answer must be the best one.
"""
import itertools

import numpy as np
import pytest

from text_embedding_encoder_gb300 import binding

UNK, BOS, EOS = 0, 1, 2
META = "▁"


@pytest.fixture(scope="module")
def lib():
    try:
        return binding.load()
    except RuntimeError:
        pytest.skip("library not built")


def _vocab(seed):
    """A small random vocabulary over a six-character alphabet (one character,
    'x', is in no piece), with pieces of one to three characters."""
    rng = np.random.default_rng(seed)
    alphabet = ["a", "b", "c", "日", "本", META]
    pieces = set(rng.choice(alphabet[:-1], 3, replace=False))      # some one-character pieces are missing
    for _ in range(25):
        k = int(rng.integers(2, 4))
        pieces.add("".join(rng.choice(alphabet, k)))
    pieces = sorted(pieces)
    # multiples of 1/8: every total is exact in float and double, so equal
    # totals are real ties and the tie rule is exercised
    scores = (-rng.integers(4, 96, len(pieces)) / 8.0).astype(np.float32)
    return ["<unk>", "<s>", "</s>"] + pieces, np.concatenate([[0.0, 0.0, 0.0], scores]).astype(np.float32)


def _brute_force(text, pieces, scores, unk_score):
    """Best-scoring segmentation by enumerating every cut of the text; among
    equal totals the documented rule: the longest last piece, then the same
    for the text before it (the piece lengths read from the end, compared
    lexicographically)."""
    text = text.replace(" ", META)
    ids = {p: i for i, p in enumerate(pieces) if i > EOS}
    m = len(text)
    best, best_key, best_ids = -np.inf, None, None
    for cuts in itertools.product([0, 1], repeat=max(0, m - 1)):
        bounds = [0] + [i + 1 for i, c in enumerate(cuts) if c] + [m]
        total, seg = 0.0, []
        for a, b in zip(bounds[:-1], bounds[1:]):
            p = text[a:b]
            if p in ids:
                total += float(scores[ids[p]])
                seg.append(ids[p])
            elif b - a == 1:
                total += unk_score
                seg.append(UNK)
            else:
                break
        else:
            key = (total, tuple(b - a for a, b in zip(bounds[:-1], bounds[1:]))[::-1])
            if best_key is None or key > best_key:
                best, best_key, best_ids = total, key, seg
    return best, best_ids


@pytest.mark.parametrize("seed", range(6))
def test_segmentation_is_the_best_by_brute_force(lib, seed):
    pieces, scores = _vocab(seed)
    tok = binding.Unigram(pieces, scores, UNK, -20.0, BOS, EOS)
    rng = np.random.default_rng(100 + seed)
    chars = ["a", "b", "c", "日", "本", " ", "x"]
    for _ in range(40):
        text = "".join(rng.choice(chars, int(rng.integers(1, 10))))
        got = tok.encode(text)
        best, want = _brute_force(text, pieces, scores, -20.0)
        assert got[0] == BOS and got[-1] == EOS
        total = sum(-20.0 if i == UNK else float(scores[i]) for i in got[1:-1])
        assert total == best, (text, got, want)
        assert got[1:-1].tolist() == want, (text, got, want)
        # the pieces put back together give the text (spaces as the meta symbol) wherever no unknown is involved
        if UNK not in got:
            assert "".join(pieces[i] for i in got[1:-1]) == text.replace(" ", META)
    tok.close()


def test_ties_prefer_the_longest_last_piece(lib):
    tok = binding.Unigram(["<unk>", "a", "b", "ab"], [0.0, -1.0, -1.0, -2.0], UNK, -10.0)
    assert tok.encode("ab").tolist() == [3]          # "ab" (-2) against "a" + "b" (-2)
    assert tok.encode("abab").tolist() == [3, 3]
    tok.close()


def test_unknown_characters_bos_eos_and_limits(lib):
    tok = binding.Unigram(["<unk>", "<s>", "</s>", "日本", "本", META + "a"], [0, 0, 0, -1.0, -2.0, -1.5],
                          UNK, -10.0, BOS, EOS)
    assert tok.encode("").tolist() == [BOS, EOS]
    assert tok.encode("日本 a").tolist() == [BOS, 3, 5, EOS]       # the space is read as U+2581
    assert tok.encode("日x本").tolist() == [BOS, UNK, UNK, 4, EOS]  # 日 alone is no piece; x is in none
    lib_ = tok.lib
    raw = "日本".encode()
    out = np.empty(2, np.int32)
    assert lib_.tee_unigram_encode(tok.h, raw, len(raw), out.ctypes.data, 2) == binding.TEE_ETOOLONG
    assert lib_.tee_unigram_encode(tok.h, b"\xff\xfe", 2, None, 0) == binding.TEE_EINVAL
    tok.close()
    no_wrap = binding.Unigram(["<unk>", "a"], [0.0, -1.0], UNK, -10.0)
    assert no_wrap.encode("aa").tolist() == [1, 1]
    no_wrap.close()


def test_bad_vocabularies_are_rejected(lib):
    for pieces, scores, unk in ((["<unk>", "a", "a"], [0, -1, -1], 0),        # duplicate piece
                                (["<unk>", ""], [0, -1], 0),                  # empty piece
                                (["<unk>", "a"], [0, float("nan")], 0),       # score not finite
                                (["<unk>", "a"], [0, -1], 5)):                # unk id out of range
        with pytest.raises(binding.TeeError) as e:
            binding.Unigram(pieces, scores, unk, -10.0)
        assert e.value.code == binding.TEE_EINVAL


def test_similarity_matrix(lib):
    rng = np.random.default_rng(3)
    v = rng.standard_normal((6, 768)).astype(np.float32)
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    sim = binding.similarity(v)
    ref = v.astype(np.float64) @ v.astype(np.float64).T
    np.testing.assert_allclose(sim, ref, atol=1e-7)
    np.testing.assert_array_equal(sim, sim.T)
    np.testing.assert_allclose(np.diag(sim), 1.0, atol=1e-6)
    text = binding.format_similarity(sim)
    lines = text.splitlines()
    assert len(lines) == 6 and all(len(ln.split()) == 6 for ln in lines)
    assert lines[0].split()[0] == "1.0000"


def test_pack_texts():
    ids, cu = binding.pack_texts([np.array([1, 5, 2]), np.array([1, 2]), np.array([1, 7, 8, 9, 2])])
    assert cu.tolist() == [0, 3, 5, 10]
    assert ids.tolist() == [1, 5, 2, 1, 2, 1, 7, 8, 9, 2]
