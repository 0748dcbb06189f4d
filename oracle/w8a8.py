"""Integer (W8A8) path of the oracle.  Test infrastructure only.

§精度と量子化 of the tensai page "テキスト埋め込み" describes the -q8 path:
the stored weight blocks are used unchanged, and the integer matrix product
also rounds the activations, one scale per row, to 7 bits.

Readings (the page fixes no formulas):
* activations: per row s = max|x| / 63 and q = clamp(rint(x / s), -63, 63)
  (round half to even); a row of zeros gives s = 0 and q = 0.
* weights: blocks of 32 consecutive input (K) elements, each with one scale
  d = max|w| / 127 and q = clamp(rint(w / d), -127, 127).
* product: per block b the exact integer sum I[m, n, b] = sum_k qa * qw, then
  y[m, n] = s_m * sum_b d[n, b] * I[m, n, b].

The -q4 path of the same section repacks the file's 4- and 6-bit block formats
unchanged; the page names those formats but does not define them.  Reading:
4- and 6-bit analogues of the 8-bit blocks defined here -- blocks of 32 K
elements, d = max|w| / L, q = clamp(rint(w / d), -L, L) with L = 7 (variant
"w4a8") or L = 31 (variant "w6a8") -- with the same 7-bit activations and the
same exact block sums.  A file of the -q4 kind mixes the two widths; each
variant here uses one width for every projection.

The quantisers decide integers from floating point, so they compute in fp32
(IEEE division, round-half-even), the precision of the device kernels; the
integer sums are exact (int64); the final combination is fp64.
"""
import numpy as np

ACT_LEVELS = 63
WEIGHT_LEVELS = 127
WEIGHT_LEVELS_4 = 7
WEIGHT_LEVELS_6 = 31
BLOCK = 32


def quantize_rows7(x):
    """Per-row 7-bit quantisation of an activation matrix [M, K] (fp32 arithmetic).

    Returns (q int8[M, K], s float32[M]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax / np.float32(ACT_LEVELS)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint(x / safe[:, None]).astype(np.float32)
    q = np.clip(q, -ACT_LEVELS, ACT_LEVELS)
    q = np.where(s[:, None] > 0, q, np.float32(0.0))
    return q.astype(np.int8), s


def quantize_weight_blocks(w, levels: int = WEIGHT_LEVELS):
    """Blockwise quantisation of a weight matrix [N, K], K a multiple of 32,
    to integers in [-levels, levels] (127: int8 blocks; 31: 6-bit; 7: 4-bit).

    Returns (q int8[N, K], d float32[N, K/32]).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = w.reshape(N, K // BLOCK, BLOCK)
    d = (np.abs(blocks).max(axis=2) / np.float32(levels)).astype(np.float32)
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    q = np.rint(blocks / safe[:, :, None]).astype(np.float32)
    q = np.clip(q, -levels, levels)
    q = np.where(d[:, :, None] > 0, q, np.float32(0.0))
    return q.reshape(N, K).astype(np.int8), d


def quantize_weight_blocks4(w):
    """4-bit blocks (the -q4 reading): codes in [-7, 7], d = max|w| / 7 per block of 32."""
    return quantize_weight_blocks(w, WEIGHT_LEVELS_4)


def quantize_weight_blocks6(w):
    """6-bit blocks (the -q4 reading): codes in [-31, 31], d = max|w| / 31 per block of 32."""
    return quantize_weight_blocks(w, WEIGHT_LEVELS_6)


def _block_product(qa, qw, b) -> np.ndarray:
    """Exact integer sum over K block b, as an fp64 array of integers.

    Every term is an integer of magnitude <= 63 * 127 and a block holds 32 of
    them, so each sum is below 2**18 in magnitude: fp64 represents it, and
    every partial sum, exactly, whatever the summation order.
    """
    sl = slice(b * BLOCK, (b + 1) * BLOCK)
    return np.asarray(qa[:, sl], np.float64) @ np.asarray(qw[:, sl], np.float64).T


def int_block_partials(qa, qw) -> np.ndarray:
    """Exact per-block integer sums I[m, n, b] = sum_{k in block b} qa[m,k] qw[n,k] (int64)."""
    qa = np.asarray(qa)
    qw = np.asarray(qw)
    M, K = qa.shape
    N = qw.shape[0]
    nb = K // BLOCK
    out = np.empty((M, N, nb), dtype=np.int64)
    for b in range(nb):
        out[:, :, b] = _block_product(qa, qw, b).astype(np.int64)
    return out


def w8a8_linear(x, qw, d) -> np.ndarray:
    """y = x W^T through the integer procedure; x is rounded to fp32 first."""
    qa, s = quantize_rows7(np.asarray(x, dtype=np.float64).astype(np.float32))
    d = np.asarray(d, dtype=np.float64)
    combined = np.zeros((qa.shape[0], qw.shape[0]), dtype=np.float64)
    for b in range(qa.shape[1] // BLOCK):
        combined += _block_product(qa, qw, b) * d[None, :, b]
    return s.astype(np.float64)[:, None] * combined
