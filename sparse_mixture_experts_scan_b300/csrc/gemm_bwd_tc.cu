// gemm_bwd_tc.cu -- the grouped GEMMs of the backward pass on the 5th-generation
// tensor core (bf16 operands, fp32 TMEM accumulators).
//
// The backward of an expert's two layers ("混合专家模型MoE入门实战" §3.2 MLP,
// trained end to end in §3.5) needs products the forward never forms:
//   dgrad (MODE rows):   dH = dYp W2_e,  dXp = dZ1 W1_e (+ dZ3 W3_e)
//       A = activation gradients, K-major (rows of the expert segment);
//       B = the weights read along their output dimension: MN-major.
//   wgrad (MODE reduce): dW2_e = dYp_e^T H_e,  dW1_e = dZ1_e^T Xp_e (dW3_e from dZ3)
//       the reduction runs over the rows (tokens) of expert e's segment, so both
//       operands are MN-major tiles of row-major activation buffers.
// An MN-major operand is loaded by TMA as boxes of 64 contiguous elements (128 B,
// 128-byte swizzle) by 64 K-rows and described to tcgen05.mma with the MN-major
// bits of the instruction descriptor (sdesc_mnmajor_sw128 for the layout).
//
// Structure as in the forward kernel: one persistent CTA per SM, warp 0 TMA,
// warp 1 tcgen05.mma (M = 128, N = 256, K = 16) into two TMEM accumulators,
// warps 2-5 epilogue.  Epilogues: bf16 store; the activation backward fused into
// dH (relu mask from the saved output, GELU from the recomputed pre-activation,
// SwiGLU pair dz1 = dh z3 silu'(z1), dz3 = dh silu(z1), in place).  In rows mode
// the act-backward epilogue writes zeros on the pad rows of a segment, so the
// wgrad that follows reduces over whole 64-row K blocks of finite zeros.  The
// pre-activations come from the forward, which keeps them under training.
// Every wait is bounded; on expiry the CTA flags the error, drains and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_tile.cuh"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB: A K-major box {64, 128} or two MN boxes {64, 64}
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB: four MN boxes {64, 64}
constexpr uint32_t kMnBox = 64 * kBK * 2;    // 8 KB: one MN-major box
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr size_t kBarBytes = 256;
constexpr size_t kTableBytes = sizeof(int) * (3 * kMaxExperts + 1);
constexpr size_t kStageEpBytes = 32 * 128;  // per epilogue warp: 32 rows x 64 bf16 columns
constexpr size_t kSmem = 1024 + kStages * (size_t)kStageBytes + kBarBytes + kTableBytes + 4 * kStageEpBytes + 16;

// Raw 32 bf16 of a row (four 16-byte groups; zeros for groups at or past N).
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* row, int col0, int N, uint4 (&u)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q)
        u[q] = (col0 + q * 8 + 8 <= N) ? *reinterpret_cast<const uint4*>(row + col0 + q * 8)
                                      : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ void unpack32(const uint4 (&u)[4], float (&v)[32])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[q * 8 + 2 * i] = __uint_as_float(w[i] << 16);
            v[q * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <int MODE, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_bwd_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                  const BwdTcArgs args)
{
    constexpr bool A_MN = MODE == kBwdReduce;
    constexpr uint32_t IDESC = idesc_bf16_f32_major(kBM, kBN, A_MN, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sB = base + kStages * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_mt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + kBarBytes);
    int* s_roff = s_mt + kMaxExperts + 1;
    int* s_rows = s_roff + kMaxExperts;
    // bf16 store epilogue: per-warp staging of 32 rows x 64 columns (16-byte units
    // XOR-swizzled by row), so that the global stores write whole 128-byte lines
    uint8_t* s_ep = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(s_rows + kMaxExperts) + 15) & ~static_cast<uintptr_t>(15));

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool fixed = args.row_off == nullptr;
    const bool split = MODE == kBwdReduce && fixed && args.split_rows > 0;
    const int G = split ? ceil_div(args.fixed_rows, args.split_rows) : (fixed ? 1 : args.G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.two_seg) {
            tma_prefetch_desc(&tmA2);
            tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();  // segment tables and operands come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += kThreads) {
        if (MODE == kBwdRows)
            s_mt[i] = fixed ? (i == 0 ? 0 : ceil_div(args.fixed_rows, kBM)) : args.mtile_off[i];
        else
            s_mt[i] = i * ceil_div(args.M, kBM);
    }
    for (int i = threadIdx.x; i < G; i += kThreads) {
        if (split) {
            s_roff[i] = i * args.split_rows;
            s_rows[i] = min(args.split_rows, args.fixed_rows - i * args.split_rows);
        } else {
            s_roff[i] = fixed ? 0 : args.row_off[i];
            s_rows[i] = fixed ? args.fixed_rows : args.rows[i];
        }
    }
    __syncthreads();

    const int n_tiles = ceil_div(args.N, kBN);
    const int total = s_mt[G] * n_tiles;
    const int kb_seg = ceil_div(args.K, kBK);  // rows mode: K blocks of one product
    auto num_kb_of = [&](int g) {
        return MODE == kBwdRows ? kb_seg * (args.two_seg ? 2 : 1) : ceil_div(s_rows[g], kBK);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, filled = 0, fill_par = 0;
            bool ok = true;
            TileMap tm;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int m, n;
                tm.locate(tile, s_mt, n_tiles, m, n);
                const int g = tm.g;
                const int nkb = num_kb_of(g);
                const int bx = args.b_col0 + n * kBN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kStageBytes);
                    uint8_t* dA = sA + stage * kABytes;
                    uint8_t* dB = sB + stage * kBBytes;
                    if constexpr (MODE == kBwdRows) {
                        const int seg = kb >= kb_seg ? 1 : 0;
                        const int kk = (kb - seg * kb_seg) * kBK;
                        const int a_row = s_roff[g] + m * kBM;
                        const int b_row = (args.b_g0 + g) * args.b_rows_per_group + kk;
                        if (seg == 0) {
                            tma_load_2d(dA, &tmA, &full[stage], kk, a_row, pol_act);
#pragma unroll
                            for (int j = 0; j < kBN / 64; ++j)
                                tma_load_2d(dB + j * kMnBox, &tmB, &full[stage], bx + j * 64, b_row, pol_w);
                        } else {
                            tma_load_2d(dA, &tmA2, &full[stage], kk, a_row, pol_act);
#pragma unroll
                            for (int j = 0; j < kBN / 64; ++j)
                                tma_load_2d(dB + j * kMnBox, &tmB2, &full[stage], bx + j * 64, b_row, pol_w);
                        }
                    } else {
                        const int kr = s_roff[g] + kb * kBK;  // token rows of this K block
#pragma unroll
                        for (int j = 0; j < kBM / 64; ++j)
                            tma_load_2d(dA + j * kMnBox, &tmA, &full[stage], args.a_col0 + m * kBM + j * 64, kr,
                                        pol_act);
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_2d(dB + j * kMnBox, &tmB, &full[stage], bx + j * 64, kr, pol_act);
                    }
                    filled |= 1u << stage;
                    fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutProducer);
                *abort_flag = 1;
                for (int s = 0; s < kStages; ++s)
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
            TileMap tm;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                int m, n;
                tm.locate(tile, s_mt, n_tiles, m, n);
                const int nkb = num_kb_of(tm.g);
                const int acc = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_par ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_u32(sA + stage * kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = A_MN ? sdesc_mnmajor_sw128(a0 + k * 2048) : sdesc_kmajor_sw128(a0 + k * 32);
                        mma_bf16_ss(d_tmem, ad, sdesc_mnmajor_sw128(b0 + k * 2048), IDESC, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&tfull[acc]);  // with no K block: arrives once earlier MMAs are done
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
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(args.C);
        __nv_bfloat16* C2 = static_cast<__nv_bfloat16*>(args.C2);
        const __nv_bfloat16* E1 = static_cast<const __nv_bfloat16*>(args.e1);
        const __nv_bfloat16* E2 = static_cast<const __nv_bfloat16*>(args.e2);
        bool ok = true;
        int it = 0;
        TileMap tm;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            int m, n;
            tm.locate(tile, s_mt, n_tiles, m, n);
            const int g = tm.g;
            const int acc = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            const bool have_k = num_kb_of(g) > 0;
            const int row = m * kBM + r_in_tile;
            long long off;    // element offset of (row, column 0) in C (and e1, e2, C2)
            bool store, zero;  // write this row; write it as zeros
            if constexpr (MODE == kBwdRows) {
                off = (long long)(s_roff[g] + row) * args.ldc;
                const bool valid = row < s_rows[g];
                // pad rows of a routed segment get zeros from the act backward
                store = valid || (EPI != kEpiStore && EPI != kEpiStoreF32 && !fixed);
                zero = !valid;
            } else {
                off = (long long)(args.c_g0 + g) * args.c_gs + (long long)row * args.ldc;
                store = row < args.M;
                zero = !have_k;
            }
            // activation backward: the saved activations of the first 32 columns are
            // fetched while the accumulator is still being computed
            constexpr bool ACT_BWD = EPI == kEpiReluBwd || EPI == kEpiGeluTanhBwd || EPI == kEpiGeluErfBwd ||
                                     EPI == kEpiSwigluBwd;
            const bool fetch = ACT_BWD && store && !zero;
            uint4 pa[4], pb[4];
            if constexpr (ACT_BWD) {
                if (fetch) {
                    load_raw32(E1 + off, n * kBN, args.N, pa);
                    if constexpr (EPI == kEpiSwigluBwd) load_raw32(E2 + off, n * kBN, args.N, pb);
                }
            }
            if (!mbar_wait(&tfull[acc], acc_par, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t t_lane = tmem_base + acc * kBN + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (EPI == kEpiStore) {
                uint8_t* stg = s_ep + q * kStageEpBytes;
                // the output row of staged row rr (0..31 of this warp) and whether it is written
                const int row_base = m * kBM + q * 32;
#pragma unroll 1
                for (int c2 = 0; c2 < kBN / 64; ++c2) {
                    uint4 u[8];
                    if (have_k) {
                        uint32_t ra[32], rb[32];
                        tmem_ld_32cols(t_lane + c2 * 64, ra);
                        tmem_ld_32cols(t_lane + c2 * 64 + 32, rb);
                        tmem_ld_wait();
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const float* fa = reinterpret_cast<const float*>(ra) + w * 8;
                            const float* fb = reinterpret_cast<const float*>(rb) + w * 8;
                            u[w] = zero ? make_uint4(0u, 0u, 0u, 0u)
                                        : make_uint4(pack_bf16x2(fa[0], fa[1]), pack_bf16x2(fa[2], fa[3]),
                                                     pack_bf16x2(fa[4], fa[5]), pack_bf16x2(fa[6], fa[7]));
                            u[4 + w] = zero ? make_uint4(0u, 0u, 0u, 0u)
                                            : make_uint4(pack_bf16x2(fb[0], fb[1]), pack_bf16x2(fb[2], fb[3]),
                                                         pack_bf16x2(fb[4], fb[5]), pack_bf16x2(fb[6], fb[7]));
                        }
                    } else {
#pragma unroll
                        for (int w = 0; w < 8; ++w) u[w] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();  // the previous pass's reads of the staging rows are done
                    uint4* srow = reinterpret_cast<uint4*>(stg + lane * 128);
#pragma unroll
                    for (int w = 0; w < 8; ++w) srow[w ^ (lane & 7)] = u[w];
                    __syncwarp();
                    const int unit = lane & 7;
                    const int col = n * kBN + c2 * 64 + unit * 8;
#pragma unroll
                    for (int it2 = 0; it2 < 8; ++it2) {
                        const int rr = it2 * 4 + (lane >> 3);
                        const int orow = row_base + rr;
                        long long o2;
                        bool ok_row;
                        if constexpr (MODE == kBwdRows) {
                            ok_row = orow < s_rows[g];
                            o2 = (long long)(s_roff[g] + orow) * args.ldc;
                        } else {
                            ok_row = orow < args.M;
                            o2 = (long long)(args.c_g0 + g) * args.c_gs + (long long)orow * args.ldc;
                        }
                        const uint4 val = reinterpret_cast<const uint4*>(stg + rr * 128)[unit ^ (rr & 7)];
                        if (ok_row && col + 8 <= args.N) *reinterpret_cast<uint4*>(C + o2 + col) = val;
                    }
                }
            } else if constexpr (EPI == kEpiStoreF32) {
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    const int col0 = n * kBN + c * 32;
                    float v[32];
                    if (have_k) {
                        uint32_t r[32];
                        tmem_ld_32cols(t_lane + c * 32, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = zero ? 0.0f : __uint_as_float(r[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                    }
                    if (!store || col0 >= args.N) continue;
                    float* crow = static_cast<float*>(args.C) + off;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        if (col0 + q4 * 4 + 4 <= args.N)
                            *reinterpret_cast<float4*>(crow + col0 + q4 * 4) =
                                make_float4(v[q4 * 4], v[q4 * 4 + 1], v[q4 * 4 + 2], v[q4 * 4 + 3]);
                }
            } else {
                // activation backward (rows mode): the accumulator holds dH
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    const int col0 = n * kBN + c * 32;
                    uint32_t r[32];
                    tmem_ld_32cols(t_lane + c * 32, r);
                    uint4 qa[4], qb[4];  // the next chunk's saved activations, in flight meanwhile
                    if (fetch && c + 1 < kBN / 32) {
                        load_raw32(E1 + off, col0 + 32, args.N, qa);
                        if constexpr (EPI == kEpiSwigluBwd) load_raw32(E2 + off, col0 + 32, args.N, qb);
                    }
                    tmem_ld_wait();
                    if (store && col0 < args.N) {
                        float v[32];
                        if (zero) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                            store_row32(C + off, col0, args.N, v);
                            if constexpr (EPI == kEpiSwigluBwd) store_row32(C2 + off, col0, args.N, v);
                        } else if constexpr (EPI == kEpiSwigluBwd) {
                            // dz1 = dh z3 silu'(z1), dz3 = dh silu(z1) (fast exp and divide: the
                            // results are rounded to bf16)
                            float z1[32], z3[32], o3[32];
                            unpack32(pa, z1);
                            unpack32(pb, z3);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float dh = __uint_as_float(r[i]);
                                const float sg = __fdividef(1.0f, 1.0f + __expf(-z1[i]));
                                o3[i] = dh * z1[i] * sg;
                                v[i] = dh * z3[i] * sg * (1.0f + z1[i] * (1.0f - sg));
                            }
                            store_row32(C + off, col0, args.N, v);
                            store_row32(C2 + off, col0, args.N, o3);
                        } else {
                            constexpr int kGeluKind = EPI == kEpiGeluTanhBwd ? kActGeluTanh : kActGeluErf;
                            float z[32];
                            unpack32(pa, z);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float dh = __uint_as_float(r[i]);
                                if constexpr (EPI == kEpiReluBwd) v[i] = z[i] > 0.0f ? dh : 0.0f;
                                else v[i] = dh * act_grad_f32<kGeluKind>(z[i]);
                            }
                            store_row32(C + off, col0, args.N, v);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        pa[q] = qa[q];
                        pb[q] = qb[q];
                    }
                }
            }
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
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int MODE, int EPI>
cudaError_t launch_t(const CUtensorMap* maps, const BwdTcArgs& a, int grid, cudaStream_t st, bool pdl)
{
    auto kern = k_gemm_bwd_tc<MODE, EPI>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), kSmem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), kSmem, st, pdl, maps[0], maps[1], maps[2], maps[3], a);
}

}  // namespace

cudaError_t launch_gemm_bwd_tc(const CUtensorMap* maps, const BwdTcArgs& a, int mode, int epi, int grid,
                               cudaStream_t st, bool pdl)
{
    if (mode == kBwdReduce) {
        if (epi == kEpiStoreF32) return launch_t<kBwdReduce, kEpiStoreF32>(maps, a, grid, st, pdl);
        return launch_t<kBwdReduce, kEpiStore>(maps, a, grid, st, pdl);
    }
    switch (epi) {
    case kEpiStoreF32: return launch_t<kBwdRows, kEpiStoreF32>(maps, a, grid, st, pdl);
    case kEpiStore: return launch_t<kBwdRows, kEpiStore>(maps, a, grid, st, pdl);
    case kEpiReluBwd: return launch_t<kBwdRows, kEpiReluBwd>(maps, a, grid, st, pdl);
    case kEpiGeluTanhBwd: return launch_t<kBwdRows, kEpiGeluTanhBwd>(maps, a, grid, st, pdl);
    case kEpiGeluErfBwd: return launch_t<kBwdRows, kEpiGeluErfBwd>(maps, a, grid, st, pdl);
    default: return launch_t<kBwdRows, kEpiSwigluBwd>(maps, a, grid, st, pdl);
    }
}

}  // namespace moe
