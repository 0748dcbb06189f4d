"""CPU oracle for the packed-varlen ModernBERT-style text-embedding encoder.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
package's smoke check and the benchmark's CPU-baseline leg import this
package.  The CUDA library never calls it and shares no code with it: the
two sides meet only in the seeded input generator, which holds none of the
encoder's arithmetic.

The oracle is a plain, slow, obviously-correct restatement of the encoder
described on the tensai page "テキスト埋め込み" (mattn.github.io/tensai/ja/
embeddings).  Citations in this package name that page and its sections:

* §何が動くか / エンコーダ  -- 25 layers, each a bias-free LayerNorm, 12-head
  attention with RoPE, and a GeGLU feed-forward; the first layer and every
  third layer after it attend to the whole text with RoPE base 160000, the
  others to 64 tokens before and after with base 10000.
* §何が動くか / プーリング  -- the final layer's output is averaged over the
  whole text and scaled to length 1.
* §何が動くか, packing paragraph -- several texts share one pass; positions
  restart per text and attention stays inside each text, so the vectors equal
  those of one-at-a-time encoding.
* §精度と量子化 -- the -q8 integer path: stored weight blocks unchanged,
  activations rounded per row to 7 bits with one scale.

The per-token (multi-vector) output follows the page "Les Embeddings
multimodaux dans Llama.cpp et GGUF" (jina.ai), section "Problèmes restants":
multi-vector embeddings are one linear layer over the token states.

Floating point is fp64 throughout (inputs widened from their fp32 or bf16
storage); the integer path accumulates exactly in int64.  Every function is
pinned by a test in ``tests/test_oracle_*.py`` against something other than
itself (brute force, closed forms, library routines, invariants).
"""
from .encoder import (  # noqa: F401
    layernorm,
    rope_cos_sin,
    apply_rope,
    attention_text,
    gelu,
    geglu,
    pool_l2,
    layer_is_global,
    OracleModel,
    encode_text_states,
    encode_text,
    encode_packed,
    encode_text_tokens,
    encode_packed_tokens,
)
from .precision import round_to_bf16  # noqa: F401
from .w8a8 import (  # noqa: F401
    quantize_rows7,
    quantize_weight_blocks,
    quantize_weight_blocks4,
    quantize_weight_blocks6,
    int_block_partials,
    w8a8_linear,
)
