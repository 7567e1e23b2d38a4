// ffn_fused_tc.cu -- both linear layers of the routed experts in one persistent
// tcgen05 launch.
//
// Expert FFN ("混合专家模型MoE入门实战" §3.2): H = act(Xp W1^T (+b1)) or SwiGLU, then
// Yp = H W2^T (+b2).  Running the two layers as two grouped-GEMM launches leaves
// SMs idle in the tail of each launch (the second layer of a Switch-sized layer
// has only 2.6 tiles per SM) and at the launch boundary.  Here the GEMM1 tiles and
// then the GEMM2 tiles of all experts form one tile list that CTAs claim
// dynamically (an atomic counter), so the tail of GEMM1 overlaps the start of
// GEMM2 and every SM stays busy until the last tile.
//
// Dependencies: a GEMM2 tile reads the H rows of one M-tile, written by the
// n_tiles1 GEMM1 tiles of that M-tile (possibly on other SMs).  After storing its
// rows of a GEMM1 tile, each of the 4 epilogue warps fences (generic -> async
// proxy, then GPU scope) and adds 1 to mt_done[M-tile] with release semantics;
// the producer of a GEMM2 tile waits (bounded) until mt_done reaches
// 4 * n_tiles1 with acquire loads, then fences the async proxy before its TMA
// loads of H.  Tiles are
// claimed in increasing order and GEMM1 tiles never wait, so every GEMM1 tile a
// GEMM2 tile depends on was claimed earlier by a CTA that will finish it: no
// deadlock, whatever the residency.
//
// Tile ids travel from the producer (which claims them) to the MMA issuer and the
// epilogue through a 4-entry shared-memory ring guarded by mbarriers.  The last
// CTA to finish resets the scheduler counters for the next launch.
//
// Shared experts ("MoE 混合专家模型串讲" §"共享专家隔离": always on, gate 1) join the
// same tile list when present: one group of all T token rows read straight from
// x, hidden S * d_ff (the S experts' W1 / W3 rows are consecutive, so their
// concatenation is one wider SwiGLU), and a GEMM2 whose K = S * d_ff runs over the
// S experts' W2 matrices in turn.  The list is
//     [shared GEMM1][routed GEMM1][routed GEMM2][shared GEMM2],
// so the shared rows keep the SMs busy while nothing else is ready and their GEMM2
// tiles, last, never wait.
#include "common.cuh"
#include "kernels.h"
#include "tc_tile.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kRing = 4;
constexpr uint32_t kABoxBytes = kABoxRows * kBK * 2;  // one A box: 32 rows x 128 bytes

template <int BN>
struct FCfg {
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr uint32_t A_BYTES = kBM * kBK * 2;
    static constexpr uint32_t B_BYTES = BN * kBK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr size_t BAR_BYTES = 512;
    static constexpr size_t TABLE_BYTES = sizeof(int) * (3 * kMaxExperts + 1);
    static constexpr size_t SMEM = 1024 + STAGES * (size_t)STAGE_BYTES + BAR_BYTES + TABLE_BYTES;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *p >= target (acquire), bounded like every wait of the kernel.
__device__ __forceinline__ bool wait_counter(const unsigned* p, unsigned target, volatile int* abort)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
        __nanosleep(64);
    }
}

// GEMM2 epilogue of a top-1 layer that finishes the combine in place: the row's
// expert output o = bf16(acc + b2) is what Yp would hold, and the token's output is
// y = bf16(gate * o) -- exactly the arithmetic of the combine kernel for one kept
// slot (an fp32 multiply-add from zero, one rounding).  Every thread of the warp
// must call it (tcgen05.ld is warp-collective).
template <int BN>
__device__ __forceinline__ void epilogue_direct(uint32_t t_lane, __nv_bfloat16* yrow, bool row_ok, int n0, int N,
                                                const __nv_bfloat16* bias, size_t bias_base, float gate)
{
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t va[32];
        tmem_ld_32cols(t_lane + c * 32, va);
        tmem_ld_wait();
        const int col0 = n0 + c * 32;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float z = __uint_as_float(va[i]);
            if (bias != nullptr && col0 + i < N) z += __bfloat162float(bias[bias_base + col0 + i]);
            o[i] = fmaf(gate, __bfloat162float(__float2bfloat16_rn(z)), 0.0f);
        }
        if (row_ok) store_row32(yrow, col0, N, o);
    }
}

template <int BN, int ACT1, bool SAVE>
__global__ void __launch_bounds__(kThreads, 1)
    k_ffn_fused_tc(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmAs1,
                   const __grid_constant__ CUtensorMap tmAs2, const __grid_constant__ CUtensorMap tmA1p,
                   const __grid_constant__ CUtensorMap tmA2p, const __grid_constant__ CUtensorMap tmAs1p,
                   const __grid_constant__ CUtensorMap tmAs2p, const FusedFfnArgs args)
{
    using C = FCfg<BN>;
    constexpr bool GATED = (ACT1 == kActSwiglu);
    constexpr int OUT1 = GATED ? BN / 2 : BN;  // GEMM1 output columns per tile
    constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sB = base + C::STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* ring_full = drain + 1;
    uint64_t* ring_empty = ring_full + kRing;
    volatile int* ring = reinterpret_cast<volatile int*>(ring_empty + kRing);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_mt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + C::BAR_BYTES);
    int* s_roff = s_mt + kMaxExperts + 1;
    int* s_rows = s_roff + kMaxExperts;

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&tfull[q], 1);
            mbar_init(&tempty[q], 4);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(&ring_full[r], 1);
            mbar_init(&ring_empty[r], 5);  // the MMA thread + the 4 epilogue warps
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB1);
        if (GATED) tma_prefetch_desc(&tmB3);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB2);
        tma_prefetch_desc(&tmA1p);
        tma_prefetch_desc(&tmA2p);
        if (args.S > 0) {
            tma_prefetch_desc(&tmAs1);
            tma_prefetch_desc(&tmAs2);
            tma_prefetch_desc(&tmAs1p);
            tma_prefetch_desc(&tmAs2p);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();  // tile tables, counters and Xp come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += kThreads) s_mt[i] = args.mtile_off[i];
    for (int i = threadIdx.x; i < G; i += kThreads) {
        s_roff[i] = args.row_off[i];
        s_rows[i] = args.rows[i];
    }
    __syncthreads();

    // tile list: [shared GEMM1 | routed GEMM1 | routed GEMM2 | shared GEMM2]
    const int ts1 = args.S > 0 ? args.mt_s * args.n_tiles_s1 : 0;
    const int ts2 = args.S > 0 ? args.mt_s * args.n_tiles2 : 0;
    const int o1 = ts1;                                   // first routed GEMM1 tile
    const int total1 = o1 + s_mt[G] * args.n_tiles1;     // first routed GEMM2 tile
    const int o2s = total1 + s_mt[G] * args.n_tiles2;     // first shared GEMM2 tile
    const int total = o2s + ts2;
    const int nkb1 = ceil_div(args.K1, kBK);
    const int nkb2 = ceil_div(args.K2, kBK);
    const int nkbs2 = args.S > 0 ? ceil_div(args.S * args.seg_k2, kBK) : 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, filled = 0, fill_par = 0;
            bool ok = true;
            TileMap tm1, tm2;
            for (int j = 0; ok; ++j) {
                const int slot = j % kRing;
                if (!mbar_wait(&ring_empty[slot], ((j / kRing) & 1) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                int t = (int)atomicAdd(args.tile_ctr, 1u);
                if (t >= total) t = -1;
                ring[slot] = t;
                mbar_arrive(&ring_full[slot]);
                if (t < 0) break;
                int m, n, g = 0;
                // kind: 0 shared GEMM1, 1 routed GEMM1, 2 routed GEMM2, 3 shared GEMM2
                const int kind = t < o1 ? 0 : t < total1 ? 1 : t < o2s ? 2 : 3;
                if (kind == 0 || kind == 3) {
                    const int ls = kind == 0 ? t : t - o2s;
                    m = ls % args.mt_s;
                    n = ls / args.mt_s;
                } else if (kind == 2) {
                    tm2.locate(t - total1, s_mt, args.n_tiles2, m, n);
                    g = tm2.g;
                } else {
                    tm1.locate(t - o1, s_mt, args.n_tiles1, m, n);
                    g = tm1.g;
                }
                if (kind >= 2) {
                    // H rows of this M-tile must be complete (all GEMM1 tiles of the M-tile)
                    const unsigned* ctr = kind == 2 ? &args.mt_done[s_mt[g] + m] : &args.mt_done[args.mt_s0 + m];
                    const unsigned need = 4u * (unsigned)(kind == 2 ? args.n_tiles1 : args.n_tiles_s1);
                    if (!wait_counter(ctr, need, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                }
                const int a_row = (kind == 1 || kind == 2) ? s_roff[g] + m * kBM : m * kBM;
                // a full M-tile's A is one box; with partial_a a partial one's the 32-row boxes
                // that hold valid rows (rows past them stay stale in shared memory; their
                // accumulator rows are never stored)
                const int a_valid = min(kBM, ((kind == 1 || kind == 2) ? s_rows[g] : args.shared_rows) - m * kBM);
                const int a_boxes = args.partial_a ? (a_valid + kABoxRows - 1) / kABoxRows : kBM / kABoxRows;
                const uint32_t stage_bytes = (uint32_t)a_boxes * kABoxBytes + C::B_BYTES;
                const CUtensorMap* mA = kind == 0 ? &tmAs1 : kind == 1 ? &tmA1 : kind == 2 ? &tmA2 : &tmAs2;
                const CUtensorMap* mAp = kind == 0 ? &tmAs1p : kind == 1 ? &tmA1p : kind == 2 ? &tmA2p : &tmAs2p;
                const int b_row = kind == 2 ? g * args.b2_rows_per_group + n * BN
                                  : kind == 1 ? g * args.b1_rows_per_group + n * OUT1
                                  : kind == 0 ? args.b1_row0 + n * OUT1
                                              : 0;  // shared GEMM2: per K segment below
                const int nkb = kind == 2 ? nkb2 : kind == 3 ? nkbs2 : nkb1;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    uint8_t* dA = sA + stage * C::A_BYTES;
                    uint8_t* dB = sB + stage * C::B_BYTES;
                    // each TMA names its kernel-parameter tensor map directly
                    if (a_boxes * kABoxRows == kBM) {
                        tma_load_2d(dA, mA, &full[stage], kb * kBK, a_row, pol_act);
                    } else {
                        for (int i = 0; i < a_boxes; ++i)
                            tma_load_2d(dA + i * kABoxBytes, mAp, &full[stage], kb * kBK, a_row + i * kABoxRows,
                                        pol_act);
                    }
                    if (kind == 2) {
                        tma_load_2d(dB, &tmB2, &full[stage], kb * kBK, b_row, pol_w);
                    } else if (kind == 3) {
                        // K column kb * 64 of the concatenated hidden layer: expert seg, column kc
                        const int seg = (kb * kBK) / args.seg_k2, kc = kb * kBK - seg * args.seg_k2;
                        tma_load_2d(dB, &tmB2, &full[stage], kc, (args.b2_group0 + seg) * args.b2_rows_per_group + n * BN,
                                    pol_w);
                    } else {
                        tma_load_2d(dB, &tmB1, &full[stage], kb * kBK, b_row, pol_w);
                        if (GATED) tma_load_2d(dB + C::B_BYTES / 2, &tmB3, &full[stage], kb * kBK, b_row, pol_w);
                    }
                    filled |= 1u << stage;
                    fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutProducer);
                *abort_flag = 1;
                for (int s = 0; s < C::STAGES; ++s)
                    if (((filled >> s) & 1u) && !mbar_wait_short(&full[s], (fill_par >> s) & 1u))
                        atomicOr(args.err, kErrTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                const int slot = j % kRing;
                if (!mbar_wait(&ring_full[slot], (j / kRing) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int t = ring[slot];
                if (t < 0) break;
                const int nkb = t < total1 ? nkb1 : t < o2s ? nkb2 : nkbs2;
                const int acc = it & 1;
                if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32),
                                    IDESC, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                mbar_arrive(&ring_empty[slot]);
                ++it;
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutMma);
                *abort_flag = 1;
            }
            mma_commit(drain);
            if (!mbar_wait_short(drain, 0)) atomicOr(args.err, kErrTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        const __nv_bfloat16* bias1 = static_cast<const __nv_bfloat16*>(args.bias1);
        const __nv_bfloat16* bias2 = static_cast<const __nv_bfloat16*>(args.bias2);
        bool ok = true;
        int it = 0;
        TileMap tm1, tm2;
        for (int j = 0; ok; ++j) {
            const int slot = j % kRing;
            if (!mbar_wait(&ring_full[slot], (j / kRing) & 1, abort_flag)) {
                ok = false;
                break;
            }
            const int t = ring[slot];
            if (t < 0) break;
            const int kind = t < o1 ? 0 : t < total1 ? 1 : t < o2s ? 2 : 3;
            int m, n, g = 0;
            if (kind == 0 || kind == 3) {
                const int ls = kind == 0 ? t : t - o2s;
                m = ls % args.mt_s;
                n = ls / args.mt_s;
            } else if (kind == 2) {
                tm2.locate(t - total1, s_mt, args.n_tiles2, m, n);
                g = tm2.g;
            } else {
                tm1.locate(t - o1, s_mt, args.n_tiles1, m, n);
                g = tm1.g;
            }
            const int acc = it & 1;
            if (!mbar_wait(&tfull[acc], (it >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int row = m * kBM + r_in_tile;
            const bool shared = kind == 0 || kind == 3;
            const bool row_ok = row < (shared ? args.shared_rows : s_rows[g]);
            const uint32_t t_lane = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            if (kind == 2 && args.y != nullptr) {
                // top-1 direct combine: the row's token and gate from the dispatch
                const int prow = s_roff[g] + (row_ok ? row : 0);
                const int tok = args.row_token[prow];
                const float gate = args.row_gate[prow];
                __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(args.y) + (size_t)(row_ok ? tok : 0) * args.ldy;
                epilogue_direct<BN>(t_lane, yrow, row_ok, n * BN, args.N2, bias2,
                                    (size_t)g * args.b2_rows_per_group, gate);
            } else if (kind == 2) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.yp) + (size_t)(s_roff[g] + row) * args.ldy;
                epilogue_tile<BN, kActNone>(t_lane, orow, row_ok, n * BN, args.N2, bias2,
                                            (size_t)g * args.b2_rows_per_group, 1, args.b2_rows_per_group);
            } else if (kind == 3) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.ys) + (size_t)row * args.ldy;
                epilogue_tile<BN, kActNone>(t_lane, orow, row_ok, n * BN, args.N2, nullptr, 0, 1, 0);
            } else if (kind == 1) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.h) + (size_t)(s_roff[g] + row) * args.ldh;
                const size_t zo = (size_t)(s_roff[g] + row) * args.ldh;
                epilogue_tile<BN, ACT1, SAVE>(t_lane, orow, row_ok, n * OUT1, args.N1, bias1,
                                              (size_t)g * args.b1_rows_per_group, 1, args.b1_rows_per_group,
                                              SAVE ? static_cast<__nv_bfloat16*>(args.z1) + zo : nullptr,
                                              SAVE && GATED ? static_cast<__nv_bfloat16*>(args.z3) + zo : nullptr);
            } else {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.hs) + (size_t)row * args.ldhs;
                const size_t zo = (size_t)row * args.ldhs;
                epilogue_tile<BN, ACT1, SAVE>(t_lane, orow, row_ok, n * OUT1, args.S * args.seg_k2, nullptr, 0, 1, 0,
                                              SAVE ? static_cast<__nv_bfloat16*>(args.zs1) + zo : nullptr,
                                              SAVE && GATED ? static_cast<__nv_bfloat16*>(args.zs3) + zo : nullptr);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (kind <= 1) {
                // publish this warp's 32 H rows to the GEMM2 tiles that read them: each
                // of the 4 epilogue warps adds 1, so an M-tile is complete at 4 * n_tiles1
                fence_proxy_async_global();
                __threadfence();
                __syncwarp();
                unsigned* ctr = kind == 1 ? &args.mt_done[s_mt[g] + m] : &args.mt_done[args.mt_s0 + m];
                if (lane == 0) red_release_gpu_add(ctr, 1u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring_empty[slot]);
            ++it;
        }
        if (!ok) {
            if (lane == 0) atomicOr(args.err, kErrTimeoutEpilogue);
            *abort_flag = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
    if (threadIdx.x == 0) {
        // the last CTA to finish re-arms the scheduler for the next launch
        __threadfence();
        if (atomicAdd(args.ctas_done, 1u) == gridDim.x - 1) {
            __threadfence();
            for (int i = 0; i < args.mt_max; ++i) args.mt_done[i] = 0u;
            *args.tile_ctr = 0u;
            __threadfence();
            *args.ctas_done = 0u;
        }
    }
}

template <int BN, int ACT1, bool SAVE>
cudaError_t launch_t(const CUtensorMap* maps, const FusedFfnArgs& a, int grid, cudaStream_t st, bool pdl)
{
    auto kern = k_ffn_fused_tc<BN, ACT1, SAVE>;
    const size_t smem = FCfg<BN>::SMEM;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    // without shared experts the shared-expert maps are never read: pass the routed ones
    const CUtensorMap& s1 = a.S > 0 ? maps[5] : maps[0];
    const CUtensorMap& s2 = a.S > 0 ? maps[6] : maps[0];
    const CUtensorMap& s1p = a.S > 0 ? maps[9] : maps[7];
    const CUtensorMap& s2p = a.S > 0 ? maps[10] : maps[7];
    return launch_kernel(kern, dim3(grid), dim3(kThreads), smem, st, pdl, maps[0], maps[1], maps[2], maps[3],
                         maps[4], s1, s2, maps[7], maps[8], s1p, s2p, a);
}

}  // namespace

cudaError_t launch_ffn_fused_tc(const CUtensorMap* maps, const FusedFfnArgs& a, int act1, int grid,
                                cudaStream_t st, bool pdl)
{
    // with a.z1 set (training, GELU or SwiGLU) the GEMM1 epilogue also keeps the pre-activations
    const bool save = a.z1 != nullptr;
    switch (act1) {
    case kActRelu: return launch_t<256, kActRelu, false>(maps, a, grid, st, pdl);
    case kActGeluTanh:
        return save ? launch_t<256, kActGeluTanh, true>(maps, a, grid, st, pdl)
                    : launch_t<256, kActGeluTanh, false>(maps, a, grid, st, pdl);
    case kActGeluErf:
        return save ? launch_t<256, kActGeluErf, true>(maps, a, grid, st, pdl)
                    : launch_t<256, kActGeluErf, false>(maps, a, grid, st, pdl);
    default:
        return save ? launch_t<256, kActSwiglu, true>(maps, a, grid, st, pdl)
                    : launch_t<256, kActSwiglu, false>(maps, a, grid, st, pdl);
    }
}

}  // namespace moe
