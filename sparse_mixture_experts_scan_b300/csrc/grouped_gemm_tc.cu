// grouped_gemm_tc.cu -- stage 3 of the layer on the 5th-generation tensor core.
//
// Every expert is a two-layer MLP ("混合专家模型MoE入门实战" §3.2; "MoE混合专家
// 模型原理与实战" §3.1): H = act(Xp W1^T (+b1)) or SwiGLU silu(Xp W1^T) * (Xp W3^T),
// then Yp = H W2^T (+b2).  Experts differ in how many rows they own, so the
// GEMM is grouped: one persistent kernel walks a device-built list of
// (expert, M-tile, N-tile) triples; segments are padded to 128 rows so a tile
// never straddles two experts and one 2-D TMA tensor map covers all of them.
//
// Per CTA (one per SM, 192 threads):
//   warp 0      TMA producer: A tile [128 x 64] + B tile [BN x 64] per stage,
//               128-byte swizzle, mbarrier transaction counts;
//   warp 1      allocates 2*BN TMEM columns (two fp32 accumulators) and one
//               lane issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide slice,
//               committing each stage back to the producer and each finished
//               accumulator to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld (one TMEM lane = one output row per
//               thread), bias + activation (or the SwiGLU pairing of the W1
//               and W3 halves of the accumulator), bf16 rounding, 16-byte stores.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// Every wait is bounded (common.cuh: mbar_wait); on expiry the CTA records an
// error bit, drains its in-flight copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_tile.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;

template <int BN>
struct TcCfg {
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr uint32_t A_BYTES = kBM * kBK * 2;
    static constexpr uint32_t B_BYTES = BN * kBK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr size_t BAR_BYTES = 256;
    static constexpr size_t TABLE_BYTES = sizeof(int) * (3 * kMaxExperts + 1);
    static constexpr size_t SMEM = 1024 + STAGES * (size_t)STAGE_BYTES + BAR_BYTES + TABLE_BYTES;
};

template <int BN, int ACT, bool SAVE>
__global__ void __launch_bounds__(kThreads, 1)
    k_grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmB3, const GroupedGemmArgs args)
{
    using C = TcCfg<BN>;
    constexpr bool GATED = (ACT == kActSwiglu);
    constexpr int OUT_COLS = GATED ? BN / 2 : BN;  // output columns per tile
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
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_mt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + C::BAR_BYTES);
    int* s_roff = s_mt + kMaxExperts + 1;
    int* s_rows = s_roff + kMaxExperts;

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool fixed = args.mtile_off == nullptr;
    const int G = fixed ? 1 : args.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (GATED) tma_prefetch_desc(&tmB3);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();  // the tile tables and the A operand come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += kThreads)
        s_mt[i] = fixed ? (i == 0 ? 0 : ceil_div(args.fixed_rows, kBM)) : args.mtile_off[i];
    for (int i = threadIdx.x; i < G; i += kThreads) {
        s_roff[i] = fixed ? 0 : args.row_off[i];
        s_rows[i] = fixed ? args.fixed_rows : args.rows[i];
    }
    __syncthreads();

    const int n_tiles = args.n_tiles;
    const int total = s_mt[G] * n_tiles;
    const int kb_per_seg = ceil_div(args.K, kBK);
    const int num_kb = args.k_segments * kb_per_seg;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_act = policy_evict_last();   // activations: re-read per N tile
            const uint64_t pol_w = policy_evict_first();    // weights: streamed
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_par = 0;  // per stage: ever filled / parity of last fill
            bool ok = true;
            TileMap tm;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int m, n;
                tm.locate(tile, s_mt, n_tiles, m, n);
                const int a_row = s_roff[tm.g] + m * kBM;
                const int b_n0 = n * (GATED ? BN / 2 : BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    const int sg = kb / kb_per_seg;
                    const int kk = (kb - sg * kb_per_seg) * kBK;
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d(sA + stage * C::A_BYTES, &tmA, &full[stage], sg * args.K + kk, a_row,
                                pol_act);
                    const int b_row = (args.b_group0 + tm.g + sg) * args.b_rows_per_group + b_n0;
                    uint8_t* dB = sB + stage * C::B_BYTES;
                    if (GATED) {
                        tma_load_2d(dB, &tmB, &full[stage], kk, b_row, pol_w);
                        tma_load_2d(dB + C::B_BYTES / 2, &tmB3, &full[stage], kk, b_row, pol_w);
                    } else {
                        tma_load_2d(dB, &tmB, &full[stage], kk, b_row, pol_w);
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
                // let every copy this CTA started land before its shared memory is released
                for (int s = 0; s < C::STAGES; ++s)
                    if (((filled >> s) & 1u) && !mbar_wait_short(&full[s], (fill_par >> s) & 1u))
                        atomicOr(args.err, kErrTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_par ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32),
                                    sdesc_kmajor_sw128(b0 + k * 32), IDESC, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&tfull[acc]);
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutMma);
                *abort_flag = 1;
            }
            // every MMA issued by this CTA completes before TMEM is released
            mma_commit(drain);
            if (!mbar_wait_short(drain, 0)) atomicOr(args.err, kErrTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        const int r_in_tile = q * 32 + lane;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
        const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(args.bias);
        bool ok = true;
        int it = 0;
        TileMap tm;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            int m, n;
            tm.locate(tile, s_mt, n_tiles, m, n);
            const int acc = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            if (!mbar_wait(&tfull[acc], acc_par, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int row = m * kBM + r_in_tile;
            const bool row_ok = row < s_rows[tm.g];
            __nv_bfloat16* orow = out + (size_t)(s_roff[tm.g] + row) * args.ldo;
            const uint32_t t_lane = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            const size_t zo = (size_t)(s_roff[tm.g] + row) * args.ldo;
            epilogue_tile<BN, ACT, SAVE>(t_lane, orow, row_ok, n * OUT_COLS, args.N, bias,
                                         (size_t)(args.b_group0 + tm.g) * args.b_rows_per_group, args.k_segments,
                                         args.b_rows_per_group,
                                         SAVE ? static_cast<__nv_bfloat16*>(args.z1) + zo : nullptr,
                                         SAVE && GATED ? static_cast<__nv_bfloat16*>(args.z3) + zo : nullptr);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
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
}

template <int BN, int ACT, bool SAVE = false>
cudaError_t launch_tc_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                        const GroupedGemmArgs& args, int grid, cudaStream_t st, bool pdl)
{
    auto kern = k_grouped_gemm_tc<BN, ACT, SAVE>;
    const size_t smem = TcCfg<BN>::SMEM;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), smem, st, pdl, a, b, b3, args);
}

template <int BN>
cudaError_t launch_tc_bn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                         const GroupedGemmArgs& args, int act, int grid, cudaStream_t st, bool pdl)
{
    // with args.z1 set (training) the epilogue also keeps the pre-activations
    const bool save = args.z1 != nullptr;
    switch (act) {
    case kActNone: return launch_tc_t<BN, kActNone>(a, b, b3, args, grid, st, pdl);
    case kActRelu: return launch_tc_t<BN, kActRelu>(a, b, b3, args, grid, st, pdl);
    case kActGeluTanh:
        return save ? launch_tc_t<BN, kActGeluTanh, true>(a, b, b3, args, grid, st, pdl)
                    : launch_tc_t<BN, kActGeluTanh>(a, b, b3, args, grid, st, pdl);
    case kActGeluErf:
        return save ? launch_tc_t<BN, kActGeluErf, true>(a, b, b3, args, grid, st, pdl)
                    : launch_tc_t<BN, kActGeluErf>(a, b, b3, args, grid, st, pdl);
    default:
        return save ? launch_tc_t<BN, kActSwiglu, true>(a, b, b3, args, grid, st, pdl)
                    : launch_tc_t<BN, kActSwiglu>(a, b, b3, args, grid, st, pdl);
    }
}

}  // namespace

size_t gemm_tc_smem(int bn) { return bn == 256 ? TcCfg<256>::SMEM : TcCfg<128>::SMEM; }

cudaError_t launch_gemm_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                           const GroupedGemmArgs& args, int act, int bn, int grid, cudaStream_t st, bool pdl)
{
    if (bn == 256) return launch_tc_bn<256>(a, b, b3, args, act, grid, st, pdl);
    return launch_tc_bn<128>(a, b, b3, args, act, grid, st, pdl);
}

}  // namespace moe
