// bf16 projection GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// The four projections of every layer (QKV, attention output, GeGLU input,
// feed-forward output; tensai page "テキスト埋め込み", §何が動くか / エンコーダ)
// are the only dense contractions of the pass.  C = A W^T with A [M, K] the
// token activations and W [N, K] the weights, both bf16 and K-contiguous.
//
// Design (one CTA per SM, persistent over output tiles):
//   * tile 128 x BN per CTA, K step 64 (one 128-byte swizzle atom); a
//     shared-memory ring of as many stages as fit, filled by TMA
//     (cp.async.bulk.tensor, 128B swizzle, out-of-range rows zero-filled).
//     BN = 256 for the bf16-output projections, 128 (short K) or 256 / 192
//     (long K) for the residual ones.
//   * CTA pairs (clusters of two) compute 256 x BN tiles with tcgen05
//     cta_group::2 MMAs (M=256) issued by the even CTA: each CTA stages its
//     128 rows of A and half of the weight tile, and holds its 128 accumulator
//     rows in its own tensor memory.  Row counts below two tiles, and the
//     short-K residual projection, run one CTA per tile (M=128 MMAs).
//   * warp 0 lane 0: TMA producer.  warp 1: TMEM allocator, lane 0 issues
//     tcgen05.mma (N=BN, K=16) and commits to mbarriers.  warps 2-5:
//     epilogue, each reading its 32-lane TMEM quadrant with tcgen05.ld.
//   * two TMEM accumulators (2 x BN fp32 columns) so the epilogue of one tile
//     overlaps the MMAs of the next.
//   * tiles are ordered with the N index fastest, so CTAs running at the same
//     time share their A rows in L2.
//   * epilogues fused into the store: bf16 store, fp32 residual add, RoPE on
//     the q/k columns (positions restart per text), GeGLU gate.  Outputs go
//     out through per-warp swizzled shared-memory boxes and TMA bulk tensor
//     stores; the residual is TMA-loaded into those boxes, updated in place.
//   * every mbarrier wait is bounded: after ~2 s the CTA raises an abort flag,
//     drains its in-flight copies and MMAs, frees TMEM, sets the timeout bit
//     of the status word and returns.
#include "tee_internal.cuh"
#include "gemm_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "tc_ptx.cuh"

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;

struct Params {
    void* C;
    int M, N, K;
    const int32_t* pos;
    const float* rope_cos;
    const float* rope_sin;
    int hidden;
    unsigned int* status;
};

// bf16-output epilogues stage each warp's 32 rows x 64 columns in a 4 KB
// swizzled box (two per warp) and store it with a TMA bulk tensor store.  The
// residual epilogue stages each warp's whole 32 x BN fp32 slice of the
// residual (BN/32 boxes of 32 x 32): TMA-loaded, updated in place, TMA-stored.
// Residual epilogue: 32-column staging boxes per warp (a ring over the warp's
// chunks: 4 for BN = 128, 192 and 256).
constexpr int RES_BOXES_MAX = 4;   // residual ring boxes (and barriers) per epilogue warp, at most
template <int BN>
__host__ __device__ constexpr int res_round_boxes() { return BN / 32 <= 4 ? BN / 32 : (BN == 192 ? 4 : BN / 64); }

template <int BN, int EPI>
constexpr uint32_t staging_bytes() {
    return EPI == GEMM_EPI_ADD_F32 ? 4u * res_round_boxes<BN>() * 4096u : 4u * 2u * 4096u;
}

// How CTAs share the work of a tile.
//   MODE_SINGLE: one CTA per 128 x BN tile.
//   MODE_PAIR: clusters of two compute one 256 x BN tile with tcgen05
//     cta_group::2 MMAs issued by the even CTA: each CTA holds its 128 rows of
//     A and half of the weight tile (BN/2 rows) in shared memory and its 128
//     rows of the accumulator in tensor memory.  A stage carries a third less
//     data per CTA than a single CTA's (so the ring gets more stages), and the
//     weight tile is read from L2 once per 256 rows.
constexpr int MODE_SINGLE = 0, MODE_PAIR = 2;
constexpr uint32_t SMEM_LIMIT = 227 * 1024;

template <int BN, int EPI, int MODE>
struct Smem {
    static constexpr uint32_t B_BYTES = (MODE == MODE_PAIR ? BN / 2 : BN) * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t FIXED = staging_bytes<BN, EPI>() + (2 * 8 + 5 + 4 * RES_BOXES_MAX) * 8 + 16 + 1024;
    static constexpr int STAGES_FIT = (int)((SMEM_LIMIT - FIXED) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;   // as many as fit, at most 8
    static constexpr uint32_t OUT_OFF = STAGES * STAGE_BYTES;
    static constexpr uint32_t BAR_OFF = OUT_OFF + staging_bytes<BN, EPI>();
    static constexpr uint32_t N_BARS = 2 * STAGES + 5 + 4 * RES_BOXES_MAX;   // + a residual barrier per staging box
    static constexpr uint32_t TOTAL = BAR_OFF + N_BARS * 8 + 16 + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;   // a power of two >= 2 * BN
    static_assert(TOTAL <= SMEM_LIMIT, "shared memory");
};

template <int BN, int EPI, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, Params p) {
    using S = Smem<BN, EPI, MODE>;
    constexpr bool PAIR = MODE == MODE_PAIR, CL = MODE != MODE_SINGLE;
    constexpr int CG = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    // barrier indices
    const int FULL = 0, EMPTY = S::STAGES, TFULL = 2 * S::STAGES, TEMPTY = 2 * S::STAGES + 2, MMA_DONE = 2 * S::STAGES + 4,
              RES = 2 * S::STAGES + 5;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m = (p.M + BM - 1) / BM, num_n = p.N / BN, num_k = p.K / BK;
    // work units: one tile, or (clustered) a pair of vertically adjacent tiles per cluster
    const uint32_t crank = CL ? cluster_ctarank() : 0;
    const int num_units = (CL ? (num_m + 1) / 2 : num_m) * num_n;
    const int unit0 = CL ? blockIdx.x / 2 : blockIdx.x;
    const int ustride = CL ? gridDim.x / 2 : gridDim.x;
    auto unit_m = [&](int u) { return CL ? 2 * (u / num_n) + (int)crank : u / num_n; };
    // PAIR: the even CTA's barriers that both CTAs' copies and epilogues signal
    auto lead_bar = [&](int i) { return mapa_shared(bar(i), 0); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), PAIR ? 256 : 128);   // every epilogue thread of the tile's CTAs
        }
        mbar_init(bar(MMA_DONE), 1);
        for (int w = 0; w < 4 * RES_BOXES_MAX; ++w) mbar_init(bar(RES + w), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC)) : "memory");
    }
    if (warp == 1) tmem_alloc<CG>(smem_u32(tmem_slot), S::TMEM_COLS);   // PAIR: both CTAs, collectively
    tc_fence_before();
    __syncthreads();
    if constexpr (CL) cluster_sync();   // the peer's copies and commits may target these barriers only after init
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above may overlap the previous kernel; global memory only after it completes
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t g = 0;
            uint32_t armed_parity[S::STAGES];
            bool armed[S::STAGES];
            for (int s = 0; s < S::STAGES; ++s) armed[s] = false, armed_parity[s] = 0;
            bool ok = true;
            // one CTA per tile (the short-K residual projection): A's tiles are
            // prefetched into L2 PF k-steps ahead of their staging loads, so the
            // shallower ring of this mode waits on L2 rather than DRAM (CTA
            // pairs measured no gain from it)
            constexpr int PF = S::STAGES + 4;
            constexpr bool PREFETCH = !PAIR;
            for (int u = unit0; u < num_units && ok; u += ustride) {
                const int n_t = u % num_n, m_t = unit_m(u);
                if (PREFETCH && num_k > S::STAGES)
                    for (int j = S::STAGES; j < PF && j < num_k; ++j) tma_prefetch_l2_2d(&tmA, j * BK, m_t * BM);
                for (int kb = 0; kb < num_k; ++kb, ++g) {
                    const int s = g % S::STAGES;
                    const uint32_t r = g / S::STAGES;
                    if (PREFETCH && num_k > S::STAGES && kb + PF < num_k)
                        tma_prefetch_l2_2d(&tmA, (kb + PF) * BK, m_t * BM);
                    if (!mbar_wait(bar(EMPTY + s), (r & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + s * S::STAGE_BYTES;
                    const uint32_t sb = sa + A_BYTES;
                    if constexpr (PAIR) {
                        // both CTAs' halves land on the even CTA's full barrier, which expects both
                        if (crank == 0) mbar_expect_tx(bar(FULL + s), 2 * S::STAGE_BYTES);
                        tma_load_2d_pair(sa, &tmA, kb * BK, m_t * BM, lead_bar(FULL + s));
                        tma_load_2d_pair(sb, &tmB, kb * BK, n_t * BN + (int)crank * (BN / 2), lead_bar(FULL + s));
                        if (crank == 0) {
                            armed[s] = true;
                            armed_parity[s] = r & 1;
                        }
                        continue;
                    }
                    mbar_expect_tx(bar(FULL + s), S::STAGE_BYTES);
                    tma_load_2d(sa, &tmA, kb * BK, m_t * BM, bar(FULL + s));
                    tma_load_2d(sb, &tmB, kb * BK, n_t * BN, bar(FULL + s));
                    armed[s] = true;
                    armed_parity[s] = r & 1;
                }
            }
            // no copy may still be landing in shared memory when the CTA exits
            for (int s = 0; s < S::STAGES; ++s)
                if (armed[s]) mbar_wait_drain(bar(FULL + s), armed_parity[s]);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (PAIR: the even CTA's, for both) ----------------
        if (lane == 0 && (!PAIR || crank == 0)) {
            constexpr uint32_t idesc = make_idesc(PAIR ? 2 * BM : BM, BN);
            uint32_t g = 0;
            int it = 0;
            bool ok = true;
            for (int u = unit0; u < num_units && ok; u += ustride, ++it) {
                const int acc = it & 1, use = it >> 1;
                if (!(PAIR ? mbar_wait_cluster(bar(TEMPTY + acc), (use & 1) ^ 1, abort_flag)
                           : mbar_wait(bar(TEMPTY + acc), (use & 1) ^ 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_k; ++kb, ++g) {
                    const int s = g % S::STAGES;
                    const uint32_t r = g / S::STAGES;
                    if (!(PAIR ? mbar_wait_cluster(bar(FULL + s), r & 1, abort_flag)
                               : mbar_wait(bar(FULL + s), r & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + s * S::STAGE_BYTES;
                    const uint64_t adesc = sw128_desc(sa);
                    const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        if constexpr (PAIR) mma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
                        else mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
                    }
                    if constexpr (PAIR) mma_commit_pair(bar(EMPTY + s), 0x3);   // both CTAs' stage s
                    else mma_commit(bar(EMPTY + s));
                }
                if (!ok) break;
                if constexpr (PAIR) mma_commit_pair(bar(TFULL + acc), 0x3);   // both CTAs' accumulator halves
                else mma_commit(bar(TFULL + acc));
            }
            // every MMA issued must be finished before TMEM is freed
            if constexpr (PAIR) mma_commit_pair(bar(MMA_DONE), 0x1);
            else mma_commit(bar(MMA_DONE));
            mbar_wait_drain(bar(MMA_DONE), 0);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        // a warp reads TMEM lanes [32 * (warp % 4), +32): rows of its quadrant
        const int quad = warp & 3;
        const int row_local = quad * 32 + lane;
        uint8_t* stage = smem + S::OUT_OFF + (warp - 2) * 8192;   // this warp's two staging boxes
        uint32_t n_stores = 0;                                     // store groups this warp committed
        // residual epilogue: chunk g (32 columns; g counts this warp's chunks
        // over its tiles) is staged in box g % RB; lane 0 issues its load RB - 1
        // chunks ahead, as soon as the store that last used the box has read it
        constexpr int RB = res_round_boxes<BN>();
        constexpr int NC = BN / 32;
        static_assert(RB >= 2 && RB <= RES_BOXES_MAX, "a warp has RES_BOXES_MAX residual barriers and ring boxes");
        uint8_t* rslice = smem + S::OUT_OFF + (warp - 2) * RB * 4096;
        int last_issued[RES_BOXES_MAX];                            // lane 0: last chunk loaded into each box
#pragma unroll
        for (int b = 0; b < RES_BOXES_MAX; ++b) last_issued[b] = -1;
        int res_done = 0;                                          // chunks consumed by this warp
        auto res_bar = [&](int b) { return bar(RES + (warp - 2) * RES_BOXES_MAX + b); };
        auto issue_res_load = [&](int g) {                         // lane 0; box g % RB is free
            const int k = g / NC, c = g % NC;
            const int u = unit0 + k * ustride;
            if (u >= num_units) return;
            const int b = g % RB;
            mbar_expect_tx(res_bar(b), 4096);
            tma_load_2d(smem_u32(rslice + b * 4096), &tmC, (u % num_n) * BN + c * 32, unit_m(u) * BM + quad * 32,
                        res_bar(b));
            last_issued[b] = g;
        };
        // Stage 64 bf16 columns of this warp's 32 rows and store them at (x, y).
        auto store64 = [&](const float* v, int x, int y) {
            uint8_t* box = stage + (n_stores & 1) * 4096;
            if (lane == 0 && n_stores >= 2) bulk_wait_read<1>();   // the box's previous store has read it
            __syncwarp();
            stage_row_bf16x64(box, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmC, smem_u32(box), x, y);
                bulk_commit();
            }
            ++n_stores;
        };
        int it = 0;
        for (int u = unit0; u < num_units; u += ustride, ++it) {
            const int acc = it & 1, use = it >> 1;
            const int n_t = u % num_n, m_t = unit_m(u);
            const int gr = m_t * BM + row_local;
            const bool valid = gr < p.M;
            const int y_box = m_t * BM + quad * 32;
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
            if constexpr (EPI == GEMM_EPI_STORE_BF16) {
                if (!mbar_wait(bar(TFULL + acc), use & 1, abort_flag)) break;
                tc_fence_after();
#pragma unroll 1
                for (int g = 0; g < BN / 64; ++g) {
                    const int col = g * 64;
                    float v[64];
                    tmem_ld64(taddr + col, v);
                    store64(v, n_t * BN + col, y_box);
                }
            } else if constexpr (EPI == GEMM_EPI_ADD_F32) {
                // this warp's 32 x BN slice of the residual, one 32-column box
                // per chunk: the box was TMA-loaded ahead of time, is updated in
                // place, TMA-stored, and then refilled with the chunk RB ahead
                if (it == 0 && lane == 0)
                    for (int g = 0; g < RB; ++g) issue_res_load(g);
                if (!mbar_wait(bar(TFULL + acc), use & 1, abort_flag)) break;
                tc_fence_after();
                bool ok = true;
                // chunk c + 1's accumulator columns are loaded from TMEM while
                // chunk c is added and stored (two register sets, loop unrolled)
                float v[2][32];
                tmem_ld32_issue(taddr, v[0]);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int g = it * NC + c;
                    const int b = g % RB;
                    if (!mbar_wait(res_bar(b), (g / RB) & 1, abort_flag)) {
                        tmem_wait_ld();
                        ok = false;
                        break;
                    }
                    res_done = g + 1;
                    tmem_wait_ld();
                    tmem_tie32(v[c & 1]);
                    if (c + 1 < NC) tmem_ld32_issue(taddr + (c + 1) * 32, v[(c + 1) & 1]);
                    uint8_t* rp = rslice + b * 4096 + lane * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float4* q = reinterpret_cast<float4*>(rp + ((k ^ (lane & 7)) << 4));
                        float4 o = *q;
                        f2_unpack(f2_add(f2_pack(o.x, o.y), f2_pack(v[c & 1][4 * k + 0], v[c & 1][4 * k + 1])), o.x, o.y);
                        f2_unpack(f2_add(f2_pack(o.z, o.w), f2_pack(v[c & 1][4 * k + 2], v[c & 1][4 * k + 3])), o.z, o.w);
                        *q = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, smem_u32(rslice + b * 4096), n_t * BN + c * 32, y_box);
                        bulk_commit();
                        if (g >= 1) {
                            bulk_wait_read<1>();           // the store of chunk g - 1 has read its box
                            issue_res_load(g - 1 + RB);
                        }
                    }
                }
                if (!ok) break;
            } else if constexpr (EPI == GEMM_EPI_ROPE_BF16) {
                // q and k tiles (columns < 2*hidden; 2*hidden is a multiple of
                // the tile width) rotate every head with the row's cos/sin,
                // fetched once per tile before the accumulator is ready
                const bool rope = n_t * BN < 2 * p.hidden;
                float cs[32], sn[32];
                if (rope) {
                    const int pos = valid ? p.pos[gr] : 0;
                    const float4* c4 = reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * 32);
                    const float4* s4 = reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 a = c4[i], b = s4[i];
                        cs[4 * i] = a.x, cs[4 * i + 1] = a.y, cs[4 * i + 2] = a.z, cs[4 * i + 3] = a.w;
                        sn[4 * i] = b.x, sn[4 * i + 1] = b.y, sn[4 * i + 2] = b.z, sn[4 * i + 3] = b.w;
                    }
                }
                if (!mbar_wait(bar(TFULL + acc), use & 1, abort_flag)) break;
                tc_fence_after();
#pragma unroll 1
                for (int hh = 0; hh < BN / 64; ++hh) {
                    const int col = hh * 64;
                    float v[64];   // one head: v[j] pairs with v[j + 32]
                    tmem_ld64(taddr + col, v);
                    if (rope) {
                        // two rotation pairs per packed fp32x2 step
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const uint64_t A = f2_pack(v[j], v[j + 1]), B = f2_pack(v[j + 32], v[j + 33]);
                            const uint64_t C = f2_pack(cs[j], cs[j + 1]);
                            f2_unpack(f2_fma(A, C, f2_mul(B, f2_pack(-sn[j], -sn[j + 1]))), v[j], v[j + 1]);
                            f2_unpack(f2_fma(B, C, f2_mul(A, f2_pack(sn[j], sn[j + 1]))), v[j + 32], v[j + 33]);
                        }
                    }
                    store64(v, n_t * BN + col, y_box);
                }
            } else {   // GEMM_EPI_GEGLU (BN == 256): columns [0, 128) GELU inputs, [128, 256) gates
                if (!mbar_wait(bar(TFULL + acc), use & 1, abort_flag)) break;
                tc_fence_after();
#pragma unroll 1
                for (int g = 0; g < BN / 128; ++g) {
                    const int col = g * 64;
                    float a[64], gt[64];
                    // both loads in flight before one wait
                    tmem_ld64_issue(taddr + col, a);
                    tmem_ld64_issue(taddr + BN / 2 + col, gt);
                    tmem_wait_ld();
                    tmem_tie64(a);
                    tmem_tie64(gt);
#pragma unroll
                    for (int j = 0; j < 64; j += 2) gelu_mul2(a[j], a[j + 1], gt[j], gt[j + 1], a[j], a[j + 1]);
                    store64(a, n_t * (BN / 2) + col, y_box);
                }
            }
            tc_fence_before();
            if constexpr (PAIR) mbar_arrive_cluster(lead_bar(TEMPTY + acc));
            else mbar_arrive(bar(TEMPTY + acc));
        }
        if (EPI == GEMM_EPI_ADD_F32 && lane == 0)   // residual loads still in flight land before exit
            for (int b = 0; b < RB; ++b)
                if (last_issued[b] >= res_done) mbar_wait_drain(res_bar(b), (last_issued[b] / RB) & 1);
        if (lane == 0) bulk_wait_all();   // stores complete before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    // PAIR: the even CTA's MMAs (which write both CTAs' tensor memory) have
    // drained before either CTA frees it
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, S::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, TEE_STATUS_TIMEOUT);
    // the peer's last copies, commits and arrivals target this CTA's barriers: leave together
    if constexpr (CL) cluster_sync();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;

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

// Output map [rows, cols] of 2- or 4-byte elements, boxes of 32 rows x 128 bytes, 128B swizzle.
bool make_out_map(CUtensorMap* map, const void* ptr, int rows, int cols, CUtensorMapDataType dt, int box_cols) {
    const int esz = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* map, const void* ptr, int rows, int K, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, int EPI, int MODE>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, const Params& p, int units,
                     int dev, int num_sms, cudaStream_t s) {
    constexpr bool CL = MODE != MODE_SINGLE;
    // per device: CTAs that can be resident at once (a multiple of 2 when
    // clustered), set together with the kernel's shared-memory attribute
    static std::mutex mu;
    static int max_grid_of[TEE_MAX_DEVICES] = {};
    constexpr uint32_t smem = Smem<BN, EPI, MODE>::TOTAL;
    auto kernel = gemm_tc_kernel<BN, EPI, MODE>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int max_grid;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!max_grid_of[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (CL) {
                int clusters = 0;
                cfg.gridDim = dim3(2 * num_sms);
                e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
                if (e != cudaSuccess) return e;
                max_grid_of[dev] = 2 * (clusters > 0 ? clusters : 1);
            } else {
                max_grid_of[dev] = num_sms;
            }
        }
        max_grid = max_grid_of[dev];
    }
    const int per_unit = CL ? 2 : 1;
    const int grid = units * per_unit < max_grid ? units * per_unit : max_grid;
    cfg.gridDim = dim3(grid);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ma, mb, mc, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

void gemm_tc_choose_tiles(int M, int N, int K, int epi, int num_sms, int* bn, int* pair) {
    const int num_m = (M + BM - 1) / BM;
    // Residual add, short K: one CTA per tile (paired CTAs wait on each
    // other's residual loads and measured slower) on 128- or 192-column tiles,
    // whichever takes fewer column-waves (waves of tiles over the SMs times the
    // tile width; the cost per column measured equal on the 310m shape), 128 on
    // a tie: at 32768 rows x 768 columns 192-column tiles fill 6.7 waves
    // instead of 10.1 and measured 4% faster; few rows keep narrow tiles so
    // more SMs work.  Residual add, long K:
    // CTA pairs on 256- or 192-column tiles, or single CTAs on 128-column
    // tiles, whichever a wave model says finishes first: waves of units over
    // the SMs (or SM pairs) times the tile width times a per-configuration
    // cost per column measured on the 310m shape (pairs on 256 columns 0.87,
    // on 192 columns 1.0, single CTAs on 128 columns 1.05).  Few rows leave
    // most SMs idle with wide pair tiles, so small batches get narrow single
    // tiles.  Other epilogues: CTA pairs on 256-column tiles where N allows
    // (GeGLU always), else 128.
    const bool add_long = epi == GEMM_EPI_ADD_F32 && K > 1024;
    int BN = epi == GEMM_EPI_ADD_F32 ? 128 : ((epi == GEMM_EPI_GEGLU || N % 256 == 0) ? 256 : 128);
    int mode = num_m >= 2 && epi != GEMM_EPI_ADD_F32 ? MODE_PAIR : MODE_SINGLE;
    auto waves = [](long units, long slots) { return (units + slots - 1) / slots; };
    if (epi == GEMM_EPI_ADD_F32 && !add_long && N % 192 == 0 &&
        waves((long)num_m * (N / 192), num_sms) * 192 < waves((long)num_m * (N / 128), num_sms) * 128)
        BN = 192;
    if (add_long) {
        const int pairs = (num_m + 1) / 2, clusters = num_sms / 2;
        double best = (double)waves((long)num_m * (N / 128), num_sms) * 128 * 1.05;
        if (num_m >= 2 && N % 256 == 0) {
            const double c = (double)waves((long)pairs * (N / 256), clusters) * 256 * 0.87;
            if (c < best) best = c, BN = 256, mode = MODE_PAIR;
        }
        if (num_m >= 2 && N % 192 == 0) {
            const double c = (double)waves((long)pairs * (N / 192), clusters) * 192 * 1.0;
            if (c < best) best = c, BN = 192, mode = MODE_PAIR;
        }
    }
    *bn = BN;
    *pair = mode == MODE_PAIR;
}

cudaError_t launch_gemm_tc(const GemmTcArgs& a, cudaStream_t s) {
    std::call_once(g_once, init_once);
    if (g_init_err != cudaSuccess) return g_init_err;
    if (a.M < 0 || a.N <= 0 || a.K <= 0 || a.N % 128 || a.K % BK) return cudaErrorInvalidValue;
    if (a.epi == GEMM_EPI_GEGLU && a.N % 256) return cudaErrorInvalidValue;
    if (a.epi < GEMM_EPI_STORE_BF16 || a.epi > GEMM_EPI_GEGLU) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.W) | reinterpret_cast<uintptr_t>(a.C)) & 15)
        return cudaErrorMisalignedAddress;
    if (a.M == 0) return cudaSuccess;
    int dev = 0, num_sms = 0;
    cudaError_t de = tee_current_device(&dev, &num_sms);
    if (de != cudaSuccess) return de;
    const int num_m = (a.M + BM - 1) / BM;
    int BN = 128, pair = 0;
    gemm_tc_choose_tiles(a.M, a.N, a.K, a.epi, num_sms, &BN, &pair);
    const int mode = pair ? MODE_PAIR : MODE_SINGLE;
    const int b_rows = mode == MODE_SINGLE ? BN : BN / 2;
    CUtensorMap ma, mb, mc_map;
    if (!make_map(&ma, a.A, a.M, a.K, BM) || !make_map(&mb, a.W, a.N, a.K, b_rows)) return cudaErrorInvalidValue;
    if (a.epi == GEMM_EPI_ADD_F32) {
        if (!make_out_map(&mc_map, a.C, a.M, a.N, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32)) return cudaErrorInvalidValue;
    } else if (!make_out_map(&mc_map, a.C, a.M, a.epi == GEMM_EPI_GEGLU ? a.N / 2 : a.N,
                             CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64)) {
        return cudaErrorInvalidValue;
    }
    Params p{a.C, a.M, a.N, a.K, a.pos, a.rope_cos, a.rope_sin, a.hidden, a.status};
    const int units = (mode != MODE_SINGLE ? (num_m + 1) / 2 : num_m) * (a.N / BN);
#define TEE_GEMM_DISPATCH(BN_, EPI_)                                                                  \
    return mode == MODE_PAIR ? launch_t<BN_, EPI_, MODE_PAIR>(ma, mb, mc_map, p, units, dev, num_sms, s)  \
                             : launch_t<BN_, EPI_, MODE_SINGLE>(ma, mb, mc_map, p, units, dev, num_sms, s)
    if (a.epi == GEMM_EPI_ADD_F32 && BN == 256) TEE_GEMM_DISPATCH(256, GEMM_EPI_ADD_F32);
    if (a.epi == GEMM_EPI_ADD_F32 && BN == 192) TEE_GEMM_DISPATCH(192, GEMM_EPI_ADD_F32);
    if (BN == 256) {
        switch (a.epi) {
            case GEMM_EPI_STORE_BF16: TEE_GEMM_DISPATCH(256, GEMM_EPI_STORE_BF16);
            case GEMM_EPI_ROPE_BF16: TEE_GEMM_DISPATCH(256, GEMM_EPI_ROPE_BF16);
            default: TEE_GEMM_DISPATCH(256, GEMM_EPI_GEGLU);
        }
    }
    switch (a.epi) {
        case GEMM_EPI_STORE_BF16: TEE_GEMM_DISPATCH(128, GEMM_EPI_STORE_BF16);
        case GEMM_EPI_ADD_F32: TEE_GEMM_DISPATCH(128, GEMM_EPI_ADD_F32);
        default: TEE_GEMM_DISPATCH(128, GEMM_EPI_ROPE_BF16);
    }
#undef TEE_GEMM_DISPATCH
}
