// Host-side front end of the encoder: Unigram segmentation of a text into
// vocabulary pieces, and the similarity matrix of unit vectors.
//
// tensai page "テキスト埋め込み", §何が動くか (トークン化): the vocabulary is a
// SentencePiece Unigram model; the text is split into the pieces whose scores
// add up to the largest total, and the ids are wrapped in <s> ... </s>; no
// space is put in front of the text.  The page's introduction: `-sim` prints
// the matrix of dot products of the unit vectors, which are their cosines.
//
// Readings where the page is silent:
//   - segmentation works on whole UTF-8 characters; a space (U+0020) is read as
//     the meta symbol U+2581 that SentencePiece vocabularies use for it, and no
//     other normalisation is applied;
//   - a character that no piece of length one covers becomes the unknown piece
//     on its own, with its own score (a piece may still cover it inside a
//     longer match);
//   - among segmentations with equal totals, the one whose last piece is the
//     longest wins, then recursively for the text before it (the search visits
//     longer last pieces first and keeps only strictly better totals).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "tee.h"
#include "tee_frontend.h"

int tee_set_global_error(int code, const char* msg);

struct tee_unigram {
    std::unordered_map<std::string, int> piece_id;
    std::vector<float> score;
    int max_chars = 1;   // longest piece, in characters
    int unk_id = 0;
    float unk_score = 0.f;
    int bos_id = -1, eos_id = -1;
};

namespace {

// Byte length of the UTF-8 character starting at s[i] (n bytes available), or
// 0 if the bytes there are not a well-formed character.
int utf8_len(const unsigned char* s, int i, int n) {
    const unsigned c = s[i];
    int len = c < 0x80 ? 1 : (c >> 5) == 0x6 ? 2 : (c >> 4) == 0xE ? 3 : (c >> 3) == 0x1E ? 4 : 0;
    if (!len || i + len > n) return 0;
    for (int k = 1; k < len; ++k)
        if ((s[i + k] & 0xC0) != 0x80) return 0;
    return len;
}

// Character boundaries of a UTF-8 string (byte offsets, first 0, last n); false if malformed.
bool char_bounds(const char* text, int n, std::vector<int>& at) {
    at.clear();
    at.push_back(0);
    const unsigned char* s = reinterpret_cast<const unsigned char*>(text);
    for (int i = 0; i < n;) {
        const int len = utf8_len(s, i, n);
        if (!len) return false;
        i += len;
        at.push_back(i);
    }
    return true;
}

// The text with every U+0020 replaced by U+2581 (E2 96 81).
std::string escape_spaces(const char* text, int n) {
    std::string out;
    out.reserve((size_t)n + 8);
    for (int i = 0; i < n; ++i) {
        if (text[i] == ' ') out += "\xE2\x96\x81";
        else out += text[i];
    }
    return out;
}

}  // namespace

extern "C" {

int tee_unigram_create(const char* const* pieces, const float* scores, int n_pieces, int unk_id, float unk_score,
                       int bos_id, int eos_id, tee_unigram** out) {
    if (!out) return tee_set_global_error(TEE_EINVAL, "unigram: out is NULL");
    *out = nullptr;
    if (!pieces || !scores || n_pieces < 1) return tee_set_global_error(TEE_EINVAL, "unigram: empty vocabulary");
    if (unk_id < 0 || unk_id >= n_pieces) return tee_set_global_error(TEE_EINVAL, "unigram: unk_id out of range");
    if (bos_id < -1 || bos_id >= n_pieces || eos_id < -1 || eos_id >= n_pieces)
        return tee_set_global_error(TEE_EINVAL, "unigram: bos_id / eos_id out of range");
    if (!isfinite(unk_score)) return tee_set_global_error(TEE_EINVAL, "unigram: unk_score must be finite");
    tee_unigram* t = new (std::nothrow) tee_unigram();
    if (!t) return tee_set_global_error(TEE_ENOMEM, "unigram: host allocation failed");
    t->score.assign(scores, scores + n_pieces);
    t->unk_id = unk_id;
    t->unk_score = unk_score;
    t->bos_id = bos_id;
    t->eos_id = eos_id;
    std::vector<int> at;
    for (int i = 0; i < n_pieces; ++i) {
        if (!pieces[i]) {
            delete t;
            return tee_set_global_error(TEE_EINVAL, "unigram: a piece is NULL");
        }
        if (!isfinite(scores[i])) {
            delete t;
            return tee_set_global_error(TEE_EINVAL, "unigram: a score is not finite");
        }
        // the unknown, BOS and EOS pieces are never matched against text
        if (i == unk_id || i == bos_id || i == eos_id) continue;
        const int n = (int)strlen(pieces[i]);
        if (n == 0 || !char_bounds(pieces[i], n, at)) {
            delete t;
            return tee_set_global_error(TEE_EINVAL, "unigram: a piece is empty or not UTF-8");
        }
        if (!t->piece_id.emplace(std::string(pieces[i], n), i).second) {
            delete t;
            return tee_set_global_error(TEE_EINVAL, "unigram: duplicate piece");
        }
        if ((int)at.size() - 1 > t->max_chars) t->max_chars = (int)at.size() - 1;
    }
    *out = t;
    return TEE_OK;
}

int tee_unigram_encode(const tee_unigram* t, const char* text, int len, int32_t* ids, int max_ids) {
    if (!t || (!text && len > 0) || len < 0) return tee_set_global_error(TEE_EINVAL, "unigram: bad arguments");
    const std::string s = escape_spaces(text ? text : "", len);
    std::vector<int> at;
    if (!char_bounds(s.data(), (int)s.size(), at)) return tee_set_global_error(TEE_EINVAL, "unigram: text is not UTF-8");
    const int m = (int)at.size() - 1;   // characters
    // best[e]: the largest total over segmentations of characters [0, e);
    // from[e] / piece[e]: where the last piece of that segmentation starts, its id
    std::vector<double> best(m + 1, -INFINITY);
    std::vector<int> from(m + 1, -1), piece(m + 1, -1);
    best[0] = 0.0;
    for (int e = 1; e <= m; ++e) {
        for (int b = e - t->max_chars < 0 ? 0 : e - t->max_chars; b < e; ++b) {   // longest last piece first
            if (best[b] == -INFINITY) continue;
            auto it = t->piece_id.find(s.substr(at[b], at[e] - at[b]));
            if (it == t->piece_id.end()) continue;
            const double c = best[b] + (double)t->score[it->second];
            if (c > best[e]) {
                best[e] = c;
                from[e] = b;
                piece[e] = it->second;
            }
        }
        // a character no single piece covers: the unknown piece
        if (t->piece_id.find(s.substr(at[e - 1], at[e] - at[e - 1])) == t->piece_id.end()) {
            const double c = best[e - 1] + (double)t->unk_score;
            if (c > best[e]) {
                best[e] = c;
                from[e] = e - 1;
                piece[e] = t->unk_id;
            }
        }
    }
    std::vector<int32_t> rev;
    for (int e = m; e > 0; e = from[e]) rev.push_back(piece[e]);
    const int count = (int)rev.size() + (t->bos_id >= 0) + (t->eos_id >= 0);
    if (!ids) return count;
    if (count > max_ids) return tee_set_global_error(TEE_ETOOLONG, "unigram: more ids than max_ids");
    int k = 0;
    if (t->bos_id >= 0) ids[k++] = t->bos_id;
    for (auto it = rev.rbegin(); it != rev.rend(); ++it) ids[k++] = *it;
    if (t->eos_id >= 0) ids[k++] = t->eos_id;
    return count;
}

void tee_unigram_destroy(tee_unigram* t) { delete t; }

int tee_similarity(const float* vecs, int n, int dim, float* sim) {
    if (!vecs || !sim || n < 0 || dim < 1) return tee_set_global_error(TEE_EINVAL, "similarity: bad arguments");
    for (int i = 0; i < n; ++i)
        for (int j = i; j < n; ++j) {
            double acc = 0.0;
            const float* a = vecs + (size_t)i * dim;
            const float* b = vecs + (size_t)j * dim;
            for (int k = 0; k < dim; ++k) acc += (double)a[k] * (double)b[k];
            sim[(size_t)i * n + j] = sim[(size_t)j * n + i] = (float)acc;
        }
    return TEE_OK;
}

}  // extern "C"
