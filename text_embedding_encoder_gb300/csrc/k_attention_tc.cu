// Varlen bidirectional attention on the 5th-generation tensor cores (sm_103a).
//
// Method: tensai page "テキスト埋め込み", §何が動くか / エンコーダ and its packing
// paragraph: every query attends only to keys of its own text -- all of them on
// the global layers (layer 0 and every third), |i - j| <= 64 on the others --
// with scores q.k / sqrt(64) and a softmax over the allowed keys.
//
// Work unit = (128-query tile, head).  The host lists the query tiles with
// their key range [k_lo, k_hi): on global layers the tiles of each text (keys =
// the text), with consecutive texts that together span at most 128 tokens
// sharing one tile, longest first; on window layers the tiles of the packed
// sequence itself.  Where texts share a tile, every row is masked to its own
// text through the per-token text bounds row_tb.  The
// kernel is persistent: one CTA per SM walks its own list of units, which the
// host balances (longest first, each to the least-loaded CTA).  Ten warps:
//   warp 0 lane 0   TMA: each unit's Q tile (double-buffered, so the next
//                   unit's Q arrives early), then its K and V tiles (128 keys)
//                   into a KV_STAGES-deep ring, straight from the packed qkv
//                   rows;
//   warp 1          TMEM allocation; lane 0 issues S_t = Q K_t^T (M=128, N=128,
//                   K=64) into TMEM S/P buffer t % 3, and O += P_t V_t (M=128,
//                   N=64, K=128) with P read from the first 64 columns of the
//                   same buffer (the A operand, written there by the softmax
//                   over S_t) and V from shared memory as an MN-major operand
//                   (no transpose), into the unit's TMEM O buffer (two, by
//                   unit).  P V runs two tiles behind S, across unit
//                   boundaries too, so S_{t+1} is ready when the softmax
//                   finishes tile t; the MMAs of one thread run in order, so
//                   S_{t+3} overwrites buffer t % 3 only after P_t V_t read it;
//   warps 2-9       two threads per query row (a warp may read only its
//                   32-lane TMEM quadrant, so warps w and w+4 share one and
//                   split the 128 key columns, and the 64 output dimensions,
//                   in halves): one 64-column TMEM load of S, the mask as a
//                   per-row interval of visible keys (on window layers first
//                   decided for the whole warp per 32-column block: a block
//                   that no row sees is skipped, one that every row sees is
//                   not masked), the tile's row maximum
//                   exchanged through shared memory with a pair barrier, the
//                   softmax in fp32 with exp2 (scale folded into one FMA)
//                   against a reference maximum that moves only when a tile's
//                   maximum exceeds it by more than 2^8 (then that row of O is
//                   rescaled in TMEM), P as bf16 pairs stored into TMEM for the
//                   P V MMA (bf16 pairs written over the tile's first 64 S
//                   columns, once both warps of the pair have read theirs); a
//                   unit's O / l is read and stored as bf16 after the next
//                   unit's first P hand-off.
// Pipeline counters run across units; every wait is bounded.
#include "tee_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

#include "tc_ptx.cuh"

namespace {

using namespace tc;

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int HD = 64;
constexpr int KV_STAGES = 5;
constexpr int NUM_THREADS = 320;
constexpr int SM_THREADS = 256;   // softmax warps 2..9
constexpr uint32_t TILE_BYTES = BQ * HD * 2;        // Q, K or V tile: 16 KB
constexpr uint32_t OFF_Q = 0;                       // 2 Q buffers
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + KV_STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + KV_STAGES * TILE_BYTES;
// barrier indices
constexpr int SP_BUFS = 3;   // TMEM S/P buffers: tile t uses buffer t % 3
constexpr int B_QF = 0, B_QE = 2, B_KVF = 4, B_KVE = B_KVF + KV_STAGES, B_SF = B_KVE + KV_STAGES,
              B_PF = B_SF + SP_BUFS, B_OE = B_PF + SP_BUFS, B_DONE = B_OE + 2, N_BARS = B_DONE + 1;
constexpr uint32_t OFF_RED = OFF_BAR + N_BARS * 8 + 16;       // row-maximum exchange: [2 tiles][2 halves][128 rows]
constexpr uint32_t OFF_REDL = OFF_RED + 2 * 2 * 128 * 4;       // row-sum exchange: [2 units][2 halves][128 rows]
constexpr uint32_t SMEM_TOTAL = OFF_REDL + 2 * 2 * 128 * 4 + 1024;
constexpr uint32_t TMEM_COLS = 512;                 // S/P: 3 x 128 columns (by tile), O: 2 x 64 (by unit)
constexpr uint32_t TM_S = 0, TM_O = SP_BUFS * BKV;

struct AttnParams {
    const int4* slots;      // {q_start, q_len | head << 16, k_lo, k_hi} per unit, CTA after CTA
    const int* slot_off;    // CTA c takes slots slot_off[c] .. slot_off[c + 1]
    const int2* row_tb;     // per token: {start, end} of its text
    int hidden;
    int window;
    float scale_log2;       // log2(e) / sqrt(64)
    bf16* o;                // [T, hidden]
    unsigned int* status;
};

__device__ __forceinline__ int n_kv_tiles(const int4& it) { return (it.w - it.z + BKV - 1) / BKV; }

// Row maximum of columns [B, E) of a thread's 64 scores, as eight partial
// maxima (partial k over the columns = k mod 8; short dependency chains),
// three scores per max instruction.
template <int B, int E>
__device__ __forceinline__ void max8(const float* v, float* m8) {
    static_assert((E - B) % 16 == 0, "whole groups of two per partial");
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float m = fmaxf(v[B + k], v[B + k + 8]);
#pragma unroll
        for (int i = B + k + 16; i < E; i += 16) m = fmax3(m, v[i], v[i + 8]);
        m8[k] = m;
    }
}

// Eight partial row sums as four fp32x2 pairs: pair c & 3 takes columns 2c and
// 2c + 1, so partial k again sums the columns = k mod 8.
struct RowSum8 {
    uint64_t s[4];
    __device__ void zero() {
#pragma unroll
        for (int k = 0; k < 4; ++k) s[k] = 0ull;
    }
    __device__ float total() const {
        float a[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) f2_unpack(s[k], a[2 * k], a[2 * k + 1]);
        return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    }
};

// p = 2^(s * scale_log2 - m) over columns [B, E): added to the partial row
// sums and packed as bf16 pairs (pk[c] holds columns 2c, 2c + 1).
template <int B, int E>
__device__ __forceinline__ void exp_pack(float* v, uint64_t sl2x2, uint64_t negm2, RowSum8& rs, uint32_t* pk) {
#pragma unroll
    for (int c = B / 2; c < E / 2; ++c) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(v[2 * c], v[2 * c + 1]), sl2x2, negm2), a, b);
        a = ex2_approx(a);
        b = ex2_approx(b);
        rs.s[c & 3] = f2_add(rs.s[c & 3], f2_pack(a, b));
        pk[c] = pack_bf16(a, b);
    }
}

template <int B, int E>
__device__ __forceinline__ void zero_pack(uint32_t* pk) {
#pragma unroll
    for (int c = B / 2; c < E / 2; ++c) pk[c] = 0u;
}

// WINDOW: the ±window layers (per-row text bounds, 32-column block skipping);
// otherwise the global layers, whose rows all see the same keys.
template <bool WINDOW>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm, AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_QF + b), 1);
            mbar_init(bar(B_QE + b), 1);
            mbar_init(bar(B_OE + b), SM_THREADS);
        }
        for (int b = 0; b < SP_BUFS; ++b) {
            mbar_init(bar(B_SF + b), 1);
            mbar_init(bar(B_PF + b), SM_THREADS);
        }
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(bar(B_KVF + s), 1);
            mbar_init(bar(B_KVE + s), 1);
        }
        mbar_init(bar(B_DONE), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm)) : "memory");
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above may overlap the previous kernel; global memory only after it completes
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            bool q_armed[2] = {false, false}, kv_armed[KV_STAGES] = {};
            uint32_t q_par[2] = {0, 0}, kv_par[KV_STAGES] = {};
            uint32_t g = 0;   // KV tiles issued
            int ui = 0;
            bool ok = true;
            const int i0 = p.slot_off[blockIdx.x], i1 = p.slot_off[blockIdx.x + 1];
            int4 it_next = i0 < i1 ? p.slots[i0] : make_int4(0, 0, 0, 0);   // units are read one ahead
            for (int i = i0; i < i1 && ok; ++i, ++ui) {
                const int4 it = it_next;
                if (i + 1 < i1) it_next = p.slots[i + 1];
                const int head = it.y >> 16;
                const int nk = n_kv_tiles(it);
                const int qb = ui & 1;
                if (!mbar_wait(bar(B_QE + qb), ((ui >> 1) & 1) ^ 1, abort_flag)) break;
                mbar_expect_tx(bar(B_QF + qb), TILE_BYTES);
                tma_load_2d(sbase + OFF_Q + qb * TILE_BYTES, &tm, head * HD, it.x, bar(B_QF + qb));
                q_armed[qb] = true;
                q_par[qb] = (ui >> 1) & 1;
                const int xk = p.hidden + head * HD, xv = 2 * p.hidden + head * HD;
                for (int kt = 0; kt < nk; ++kt, ++g) {
                    const int s = g % KV_STAGES;
                    const uint32_t r = g / KV_STAGES;
                    if (!mbar_wait(bar(B_KVE + s), (r & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int y = it.z + kt * BKV;
                    mbar_expect_tx(bar(B_KVF + s), 2 * TILE_BYTES);
                    tma_load_2d(sbase + OFF_K + s * TILE_BYTES, &tm, xk, y, bar(B_KVF + s));
                    tma_load_2d(sbase + OFF_V + s * TILE_BYTES, &tm, xv, y, bar(B_KVF + s));
                    kv_armed[s] = true;
                    kv_par[s] = r & 1;
                }
            }
            for (int b = 0; b < 2; ++b)
                if (q_armed[b]) mbar_wait_drain(bar(B_QF + b), q_par[b]);
            for (int s = 0; s < KV_STAGES; ++s)
                if (kv_armed[s]) mbar_wait_drain(bar(B_KVF + s), kv_par[s]);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc(BQ, BKV);
            constexpr uint32_t idesc_pv = make_idesc(BQ, HD) | IDESC_B_MN_MAJOR;
            // P_tt V_tt accumulated into the unit's TMEM O buffer; the first
            // tile of a unit overwrites it once the softmax warps have read the
            // unit two back out of that buffer
            auto issue_pv = [&](uint32_t tt, bool first, int ub, uint32_t uuse) -> bool {
                const int sb = tt % SP_BUFS, st = tt % KV_STAGES;
                if (!mbar_wait(bar(B_PF + sb), (tt / SP_BUFS) & 1, abort_flag)) return false;
                if (first && !mbar_wait(bar(B_OE + ub), (uuse & 1) ^ 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t pbase = tmem_base + TM_S + sb * BKV;
                const uint32_t vbase = sbase + OFF_V + st * TILE_BYTES;
#pragma unroll
                for (int s = 0; s < BKV / 16; ++s) {
                    const uint64_t vdesc = sw128_desc_mn(vbase + s * 2048);
                    mma_bf16_ts(tmem_base + TM_O + ub * HD, pbase + 8 * s, vdesc, idesc_pv, !(first && s == 0));
                }
                // one commit frees the K/V stage and tells the softmax warps
                // that P_tt V_tt is in O
                mma_commit(bar(B_KVE + st));
                return true;
            };
            struct Pend {
                uint32_t t, use;
                bool first;
                int ub;
            };
            Pend q0{}, q1{};         // tiles whose S is issued and whose P V is not (at most two)
            int nq = 0;
            uint32_t t = 0;          // tiles whose S has been issued (global)
            bool ok = true;
            int ui = 0;
            const int i0 = p.slot_off[blockIdx.x], i1 = p.slot_off[blockIdx.x + 1];
            int4 it_next = i0 < i1 ? p.slots[i0] : make_int4(0, 0, 0, 0);
            for (int i = i0; i < i1 && ok; ++i, ++ui) {
                const int nk = n_kv_tiles(it_next);
                if (i + 1 < i1) it_next = p.slots[i + 1];
                const int qb = ui & 1;
                if (!mbar_wait(bar(B_QF + qb), (ui >> 1) & 1, abort_flag)) break;
                const uint64_t qdesc = sw128_desc(sbase + OFF_Q + qb * TILE_BYTES);
                for (int kt = 0; kt < nk; ++kt, ++t) {
                    // buffer t % 3 last held tile t - 3, whose P V was issued
                    // before this S (and runs before it): no wait for it here
                    const int st = t % KV_STAGES, sb = t % SP_BUFS;
                    if (!mbar_wait(bar(B_KVF + st), (t / KV_STAGES) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kdesc = sw128_desc(sbase + OFF_K + st * TILE_BYTES);
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k)
                        mma_bf16(tmem_base + TM_S + sb * BKV, qdesc + 2 * k, kdesc + 2 * k, idesc_s, k != 0);
                    mma_commit(bar(B_SF + sb));
                    if (kt == nk - 1) mma_commit(bar(B_QE + qb));   // Q buffer free once these S MMAs finish
                    const Pend cur{t, (uint32_t)ui >> 1, kt == 0, ui & 1};
                    if (nq == 2) {   // P V two tiles behind S
                        if (!issue_pv(q0.t, q0.first, q0.ub, q0.use)) {
                            ok = false;
                            break;
                        }
                        q0 = q1;
                        q1 = cur;
                    } else if (nq == 1) {
                        q1 = cur;
                        nq = 2;
                    } else {
                        q0 = cur;
                        nq = 1;
                    }
                }
            }
            if (ok && nq >= 1) ok = issue_pv(q0.t, q0.first, q0.ub, q0.use);
            if (ok && nq == 2) ok = issue_pv(q1.t, q1.first, q1.ub, q1.use);
            mma_commit(bar(B_DONE));
            mbar_wait_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else {
        // ---------------- softmax / output (warps 2..9) ----------------
        // Warps w and w + 4 share a TMEM lane quadrant (rows 32*quad ..) and
        // split each tile's 128 key columns; the tile's row maximum is exchanged
        // through shared memory.  P V accumulates in TMEM across the unit's key
        // tiles against a reference maximum m_ref that moves only when a tile's
        // maximum exceeds it by more than RESCALE_LOG2 (then the row of O is
        // rescaled in TMEM), so most tiles touch no O at all.
        constexpr float RESCALE_LOG2 = 8.0f;
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;               // key columns [64*half, +64), O columns [32*half, +32)
        const int r = quad * 32 + lane;                 // query row of the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float* red = reinterpret_cast<float*>(smem + OFF_RED);   // [2][2][128]
        float* red_l = reinterpret_cast<float*>(smem + OFF_REDL);   // [2][2][128]
        const uint32_t pair_bar = 1 + quad;             // named barrier of warps (w, w + 4)
        const float sl2 = p.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t t = 0;
        bool ok = true;

        auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
        // P_tt V_tt is in O once tile tt's K/V stage is released (the commit
        // after that P V).  The wait's parity cannot alias: it is asked for
        // after the S of tile tt was seen ready, and that S was issued after
        // the P V of tile tt - 3, so the stage's previous phase (tile tt - 5)
        // is complete; its next phase needs the P of tile tt + 5, which these
        // warps have not yet written.
        auto pv_done = [&](uint32_t tt) -> bool {
            return mbar_wait(bar(B_KVE + tt % KV_STAGES), (tt / KV_STAGES) & 1, abort_flag);
        };

        // The previous unit's output, deferred past the next unit's first
        // softmax: wait for its last P V, read this warp's 32 columns of O,
        // release the buffer, store O / l.  The pair's two halves of the row
        // sum l travel with the next unit's first row-maximum exchange (slot
        // by the unit's O buffer, so a slot is rewritten only after both warps
        // have passed a later exchange); the last unit exchanges them itself.
        bool pend = false;
        float l_p = 0.f, l_tot_p = 0.f;
        uint32_t t_p = 0;
        int ub_p = 0;
        bf16* dst_p = nullptr;
        auto finalize = [&](bool exchanged) -> bool {
            if (!pv_done(t_p)) return false;
            tc_fence_after();
            float o[32];
            tmem_ld32(tmem_base + lane_off + TM_O + ub_p * HD + half * 32, o);
            tc_fence_before();
            mbar_arrive(bar(B_OE + ub_p));
            if (!exchanged) {
                red_l[(ub_p * 2 + half) * 128 + r] = l_p;
                pair_sync();
                l_tot_p = l_p + red_l[(ub_p * 2 + (half ^ 1)) * 128 + r];
            }
            if (dst_p) {
                const float inv = 1.0f / l_tot_p;
#pragma unroll
                for (int d = 0; d < 32; ++d) o[d] *= inv;
                store_bf16x32(dst_p, o);
            }
            pend = false;
            return true;
        };

        // Work items are read two units ahead and the row's text bounds one
        // unit ahead, so neither load's latency lands on a unit's first tile.
        auto row_bounds = [&](const int4& x) -> int2 {
            return r < (x.y & 0xffff) ? p.row_tb[x.x + r] : make_int2(0, 0);
        };
        int ui = 0;
        const int i0 = p.slot_off[blockIdx.x], i1 = p.slot_off[blockIdx.x + 1];
        int4 it_next = i0 < i1 ? p.slots[i0] : make_int4(0, 0, 0, 0);
        int4 it_next2 = i0 + 1 < i1 ? p.slots[i0 + 1] : make_int4(0, 0, 0, 0);
        int2 tb_next = row_bounds(it_next);
        for (int i = i0; i < i1 && ok; ++i, ++ui) {
            const int4 it = it_next;
            const int2 tb = tb_next;
            it_next = it_next2;
            if (i + 1 < i1) tb_next = row_bounds(it_next);
            if (i + 2 < i1) it_next2 = p.slots[i + 2];
            const int head = it.y >> 16;
            const int q_start = it.x, q_len = it.y & 0xffff, k_lo = it.z, k_hi = it.w;
            const int nk = n_kv_tiles(it);
            const int qg = q_start + r;
            const int ub = ui & 1;
            // keys visible to this row: [vis_lo, vis_hi) -- the row's text on
            // global layers, the window inside the row's own text otherwise
            // (nothing for window rows past the end of the sequence)
            int vis_lo = k_lo, vis_hi = k_hi;
            if constexpr (WINDOW) {
                if (r < q_len) {
                    vis_lo = max(tb.x, qg - p.window);
                    vis_hi = min(tb.y, qg + p.window + 1);
                } else {
                    vis_hi = vis_lo;
                }
            } else if (r < q_len) {   // a tile shared by short texts: the row's own text
                vis_lo = max(k_lo, tb.x);
                vis_hi = min(k_hi, tb.y);
            }
            float m_ref = -INFINITY, l = 0.f;
            for (int kt = 0; kt < nk; ++kt, ++t) {
                const int sb = t % SP_BUFS;
                const int key0 = k_lo + kt * BKV + half * 64;
                const int lo = vis_lo - key0, hi = vis_hi - key0;   // visible columns [lo, hi)
                // Window layers: the warp's 64 columns as two 32-column blocks,
                // each decided for the whole warp (before S is ready: the
                // decision needs no score): no row sees a key of it (skipped:
                // no maximum, no exponentials, P = 0), every row sees all of it
                // (no mask), or a mixed block (masked per element).  The band
                // crosses one mixed block per pair of warps and tile.  Global
                // layers: every block counts as seen (a tile past the text's
                // end is masked per element).
                bool any0 = true, any1 = true, all0 = true, all1 = true;
                if constexpr (WINDOW) {
                    any0 = __any_sync(0xffffffffu, lo < hi && lo < 32 && hi > 0);
                    any1 = __any_sync(0xffffffffu, lo < hi && lo < 64 && hi > 32);
                    all0 = __all_sync(0xffffffffu, lo <= 0 && hi >= 32);
                    all1 = __all_sync(0xffffffffu, lo <= 32 && hi >= 64);
                }
                if (!mbar_wait(bar(B_SF + sb), (t / SP_BUFS) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[64];
                tmem_ld64(tmem_base + lane_off + TM_S + sb * BKV + half * 64, v);
                if constexpr (WINDOW) {
                    if (any0 && !all0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < lo || i >= hi) v[i] = -INFINITY;
                    }
                    if (any1 && !all1) {
#pragma unroll
                        for (int i = 32; i < 64; ++i)
                            if (i < lo || i >= hi) v[i] = -INFINITY;
                    }
                } else if (lo > 0 || hi < 64) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (i < lo || i >= hi) v[i] = -INFINITY;
                }
                // row maximum and (below) row sum over eight independent
                // partials: short dependency chains for the latency-bound warps
                float m8[8];
                if (any0 && any1) {
                    max8<0, 64>(v, m8);
                } else if (any0) {
                    max8<0, 32>(v, m8);
                } else if (any1) {
                    max8<32, 64>(v, m8);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
                }
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                float* red_t = red + (t & 1) * 256;
                red_t[half * 128 + r] = mx;
                const bool carry_l = kt == 0 && pend;   // the previous unit's row sum rides along
                if (carry_l) red_l[(ub_p * 2 + half) * 128 + r] = l_p;
                pair_sync();
                mx = fmaxf(mx, red_t[(half ^ 1) * 128 + r]) * sl2;
                if (carry_l) l_tot_p = l_p + red_l[(ub_p * 2 + (half ^ 1)) * 128 + r];
                if (kt == 0) {
                    m_ref = mx;
                } else {
                    // both warps of the pair see the same row maxima, so they
                    // agree on which rows (and so whether the warp) rescale
                    const bool need = mx > m_ref + RESCALE_LOG2;
                    if (__any_sync(0xffffffffu, need)) {
                        const float corr = need ? ex2_approx(m_ref - mx) : 1.0f;
                        // P V of the previous tile must be in O before it is rescaled
                        if (!pv_done(t - 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        float o[32];
                        const uint32_t oaddr = tmem_base + lane_off + TM_O + ub * HD + half * 32;
                        tmem_ld32(oaddr, o);
#pragma unroll
                        for (int d = 0; d < 32; ++d) o[d] *= corr;
                        tmem_st32(oaddr, o);
                        tc_fence_before();
                        if (need) {
                            l *= corr;
                            m_ref = mx;
                        }
                    }
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                const uint64_t negm2 = f2_pack(-m_use, -m_use);
                RowSum8 rs;
                rs.zero();
                // P as bf16 pairs over the tile's first 64 S columns (the A
                // operand of P V): this half's 64 keys are columns [32 * half,
                // +32).  Both warps of the pair have read their S (the row
                // maximum exchange above), so overwriting the other half's S
                // columns is safe.
                uint32_t pk[32];
                if (any0 && any1) {   // one loop over all 64 columns: the common case on global layers
                    exp_pack<0, 64>(v, sl2x2, negm2, rs, pk);
                } else {
                    if (any0) exp_pack<0, 32>(v, sl2x2, negm2, rs, pk);
                    else zero_pack<0, 32>(pk);
                    if (any1) exp_pack<32, 64>(v, sl2x2, negm2, rs, pk);
                    else zero_pack<32, 64>(pk);
                }
                const float sum = rs.total();
                tmem_st32_u(tmem_base + lane_off + TM_S + sb * BKV + half * 32, pk);
                tc_fence_before();
                mbar_arrive(bar(B_PF + sb));
                l += sum;
                // the previous unit's output, once this tile's P is handed over
                if (kt == 0 && pend && !finalize(true)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            l_p = l;
            t_p = t - 1;
            ub_p = ub;
            dst_p = r < q_len ? p.o + (size_t)qg * p.hidden + head * HD + half * 32 : nullptr;
            pend = true;
        }
        if (ok && pend) ok = finalize(false);
        // A warp that gave up on a bounded wait leaves with one arrival on its
        // pair barrier, so a partner already waiting there is released (and
        // next sees the abort flag at its next, bounded, wait: every path
        // between two pair barriers passes one).  Unawaited, it is harmless.
        if (!ok) asm volatile("bar.arrive %0, 64;" ::"r"(pair_bar) : "memory");
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, TEE_STATUS_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;
std::mutex g_attr_mu;
bool g_attr_set[TEE_MAX_DEVICES] = {};   // the kernel's shared-memory attribute, per device

void init_once() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        g_init_err = e != cudaSuccess ? e : cudaErrorNotSupported;
        return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t launch_attention_tc(const void* qkv, int T, int H, int n_heads, const int4* d_slots,
                                const int32_t* d_slot_off, int grid, bool is_global, int window, const int2* row_tb,
                                void* o, unsigned int* status, cudaStream_t s) {
    std::call_once(g_once, init_once);
    if (g_init_err != cudaSuccess) return g_init_err;
    if (grid == 0 || T == 0) return cudaSuccess;
    if (H != n_heads * HD || (reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(o) & 15))
        return cudaErrorInvalidValue;
    if (!row_tb || !d_slots || !d_slot_off || grid < 0) return cudaErrorInvalidValue;
    CUtensorMap tm;
    cuuint64_t dims[2] = {(cuuint64_t)3 * H, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)3 * H * 2};
    cuuint32_t box[2] = {(cuuint32_t)HD, (cuuint32_t)BQ};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    int dev = 0, num_sms = 0;
    cudaError_t de = tee_current_device(&dev, &num_sms);
    if (de != cudaSuccess) return de;
    {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        if (!g_attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)SMEM_TOTAL);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_TOTAL);
            if (e != cudaSuccess) return e;
            g_attr_set[dev] = true;
        }
    }
    AttnParams p{d_slots, d_slot_off, row_tb, H, window, 1.4426950408889634f / 8.0f, (bf16*)o, status};
    cudaError_t e = is_global ? launch_pdl(attn_tc_kernel<false>, dim3(grid), dim3(NUM_THREADS), SMEM_TOTAL, s, tm, p)
                              : launch_pdl(attn_tc_kernel<true>, dim3(grid), dim3(NUM_THREADS), SMEM_TOTAL, s, tm, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
