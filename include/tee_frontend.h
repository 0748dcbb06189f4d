/*
 * tee_frontend.h -- host-side front end of the encoder (same library as tee.h).
 *
 * Nothing here touches a GPU: these calls turn a text into the token ids the
 * encoder takes, and the encoder's unit vectors into their similarity matrix.
 * Return codes as in tee.h; messages of failed calls in tee_last_error(NULL).
 *
 * tensai page "テキスト埋め込み", §何が動くか (トークン化): the vocabulary is a
 * SentencePiece Unigram model; a text is split into the vocabulary pieces whose
 * scores add up to the largest total, and the ids are wrapped in <s> ... </s>;
 * no space is put in front of the text.  Introduction: `-sim` prints the
 * matrix of dot products of the (unit) vectors, i.e. their cosines.
 */
#ifndef TEE_FRONTEND_H
#define TEE_FRONTEND_H

#include <stdint.h>
#include "tee.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tee_unigram tee_unigram;

/*
 * Build a Unigram segmenter from a vocabulary.
 *   pieces     n_pieces NUL-terminated UTF-8 strings (host, copied); piece i has id i
 *   scores     n_pieces finite floats, the pieces' scores (log-probabilities)
 *   unk_id     id emitted for a character that no one-character piece covers,
 *              with score unk_score (finite); 0 <= unk_id < n_pieces
 *   bos_id, eos_id  ids put before / after every text, or -1 for none
 * The unk, BOS and EOS entries are never matched against text; every other
 * piece must be non-empty, valid UTF-8 and unique.  Spaces in a vocabulary
 * are written as U+2581, as SentencePiece stores them.
 * Errors: TEE_EINVAL, TEE_ENOMEM.  *out is NULL on failure.
 */
int tee_unigram_create(const char* const* pieces, const float* scores, int n_pieces, int unk_id, float unk_score,
                       int bos_id, int eos_id, tee_unigram** out);

/*
 * Segment `text` (len bytes of UTF-8, not NUL-terminated; host) into the piece
 * ids of the segmentation with the largest total score, wrapped in BOS / EOS
 * when those are set.  Every U+0020 of the text is read as U+2581; no other
 * normalisation is applied.  A character that no one-character piece covers
 * is the unknown piece on its own.  Among equal totals the segmentation whose
 * last piece is longest wins (then the same rule for the text before it).
 * ids: host int32[max_ids], or NULL to ask for the count only.
 * Returns the number of ids (>= 0), or TEE_EINVAL (not UTF-8, bad arguments),
 * TEE_ETOOLONG (more than max_ids).
 */
int tee_unigram_encode(const tee_unigram* tok, const char* text, int len, int32_t* ids, int max_ids);

/* Release a segmenter.  NULL-safe. */
void tee_unigram_destroy(tee_unigram* tok);

/*
 * Similarity matrix of n vectors: sim[i * n + j] = sum_k v_i[k] v_j[k],
 * accumulated in double and rounded to float once; symmetric by construction.
 * For the encoder's unit vectors the diagonal is 1 and each entry is a cosine.
 * vecs host float[n * dim], sim host float[n * n].  Errors: TEE_EINVAL.
 */
int tee_similarity(const float* vecs, int n, int dim, float* sim);

#ifdef __cplusplus
}
#endif
#endif /* TEE_FRONTEND_H */
