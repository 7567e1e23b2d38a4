// grouped_gemm_q8.cu -- stage 3 with int8 expert weights (bf16 activations).
//
// "MoE架构解析" §"部署实践": expert weights converted to 8-bit integers lose
// almost no accuracy and cut the bytes the HBM-bound expert stage streams;
// "MoE混合专家模型原理与实战" §"量化与PagedAttention结合": the experts are
// quantised, the router keeps its precision.  Weights are symmetric per output
// row: W[n, k] = q[n, k] * scale[n], q in [-127, 127].  An int8 value is exact in
// bf16, so the tensor core multiplies the integers themselves and
//     sum_k A[m, k] W[n, k] = scale[n] * sum_k A[m, k] q[n, k]
// lets the epilogue apply the scale once per output column, before bias and
// activation (SwiGLU: the W1 and W3 halves each with their own scale).
//
// Per CTA (one per SM, 448 threads):
//   warp 0      TMA: A tile [128 x 64] bf16 (128-byte swizzle) and the int8 B tile
//               [BN x 64] (64-byte rows, no swizzle) per stage;
//   warp 1      TMEM allocation and tcgen05.mma (M = 128, N = 256, K = 16);
//   warps 2-5   epilogue (scale, bias, activation, bf16 store);
//   warps 6-13  convert each landed int8 B tile into the bf16 K-major operand with
//               the 128-byte swizzle, fence it to the async proxy and release the
//               stage to the MMA issuer.
// Every wait is bounded (as in the bf16 kernels).
#include "common.cuh"
#include "kernels.h"
#include "tc_tile.cuh"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kThreads = 448;
constexpr int kStages = 3;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kBqBytes = kBN * kBK;        // 16 KB int8
constexpr uint32_t kBbBytes = kBN * kBK * 2;    // 32 KB bf16
constexpr uint32_t kTxBytes = kABytes + kBqBytes;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr size_t kBarBytes = 256;
constexpr size_t kTableBytes = sizeof(int) * (3 * kMaxExperts + 1);
constexpr size_t kSmem = 1024 + kStages * (size_t)(kABytes + kBqBytes + kBbBytes) + kBarBytes + kTableBytes;

// int8 x 8 (two 32-bit words) -> bf16 x 8 (one 16-byte group), exactly, without
// integer-to-float conversions: flipping the sign bit turns v into the byte v + 128,
// which a byte permute places in the low mantissa of 2^23 (0x4B0000uu); subtracting
// 2^23 + 128 leaves v exactly in fp32, and |v| <= 128 is exact in bf16.
__device__ __forceinline__ uint32_t i8pair_to_bf16x2(uint32_t u, uint32_t sel_lo, uint32_t sel_hi)
{
    const float lo = __uint_as_float(__byte_perm(u, 0x4B000000u, sel_lo)) - 8388736.0f;
    const float hi = __uint_as_float(__byte_perm(u, 0x4B000000u, sel_hi)) - 8388736.0f;
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ uint4 i8x8_to_bf16(uint2 w)
{
    const uint32_t a = w.x ^ 0x80808080u, b = w.y ^ 0x80808080u;
    // selector 0x754k: byte k of u, then 0x00, 0x00, 0x4B (bytes 4, 5, 7 of the constant)
    return make_uint4(i8pair_to_bf16x2(a, 0x7540u, 0x7541u), i8pair_to_bf16x2(a, 0x7542u, 0x7543u),
                      i8pair_to_bf16x2(b, 0x7540u, 0x7541u), i8pair_to_bf16x2(b, 0x7542u, 0x7543u));
}

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Epilogue of one accumulator row: out = act(scale * acc (+ bias)), or SwiGLU of
// the scaled W1 and W3 halves.  Scales (and bias) of output column c are at
// [col_base + c] (W3 half: scale3).  Warp-collective (tcgen05.ld).
template <int ACT>
__device__ __forceinline__ void epilogue_q8(uint32_t t_lane, __nv_bfloat16* orow, bool row_ok, int n0, int N,
                                            const float* scale, const float* scale3, const __nv_bfloat16* bias)
{
    constexpr bool GATED = (ACT == kActSwiglu);
    constexpr int OUT_COLS = GATED ? kBN / 2 : kBN;
#pragma unroll 1
    for (int c = 0; c < OUT_COLS / 32; ++c) {
        const int col0 = n0 + c * 32;
        uint32_t va[32], vb[32];
        tmem_ld_32cols(t_lane + c * 32, va);
        if constexpr (GATED) tmem_ld_32cols(t_lane + kBN / 2 + c * 32, vb);
        tmem_ld_wait();
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int col = col0 + i < N ? col0 + i : N - 1;  // clamp: columns >= N are not stored
            float z = __uint_as_float(va[i]) * scale[col];
            if constexpr (GATED) {
                o[i] = activate_bf16out<kActSwiglu>(z) * (__uint_as_float(vb[i]) * scale3[col]);
            } else {
                if (bias != nullptr) z += __bfloat162float(bias[col]);
                o[i] = activate_bf16out<ACT>(z);
            }
        }
        if (row_ok) store_row32(orow, col0, N, o);
    }
}

template <int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    k_grouped_gemm_q8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmQ3, const GroupedGemmQ8Args args)
{
    constexpr bool GATED = (ACT == kActSwiglu);
    constexpr int OUT_COLS = GATED ? kBN / 2 : kBN;
    constexpr uint32_t IDESC = idesc_bf16_f32(kBM, kBN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sBb = sA + kStages * kABytes;
    uint8_t* sBq = sBb + kStages * kBbBytes;
    uint64_t* full_q = reinterpret_cast<uint64_t*>(sBq + kStages * kBqBytes);
    uint64_t* full_b = full_q + kStages;
    uint64_t* empty = full_b + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_mt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full_q) + kBarBytes);
    int* s_roff = s_mt + kMaxExperts + 1;
    int* s_rows = s_roff + kMaxExperts;

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_q[s], 1);
            mbar_init(&full_b[s], 8);  // one arrival per converter warp
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
        tma_prefetch_desc(&tmQ);
        if (GATED) tma_prefetch_desc(&tmQ3);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();  // tile tables and A come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += kThreads) s_mt[i] = args.mtile_off[i];
    for (int i = threadIdx.x; i < G; i += kThreads) {
        s_roff[i] = args.row_off[i];
        s_rows[i] = args.rows[i];
    }
    __syncthreads();

    const int n_tiles = args.n_tiles;
    const int total = s_mt[G] * n_tiles;
    const int num_kb = ceil_div(args.K, kBK);

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
                const int a_row = s_roff[tm.g] + m * kBM;
                const int b_row = tm.g * args.b_rows_per_group + n * OUT_COLS;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_q[stage], kTxBytes);
                    tma_load_2d(sA + stage * kABytes, &tmA, &full_q[stage], kb * kBK, a_row, pol_act);
                    uint8_t* dq = sBq + stage * kBqBytes;
                    if (GATED) {
                        tma_load_2d(dq, &tmQ, &full_q[stage], kb * kBK, b_row, pol_w);
                        tma_load_2d(dq + kBqBytes / 2, &tmQ3, &full_q[stage], kb * kBK, b_row, pol_w);
                    } else {
                        tma_load_2d(dq, &tmQ, &full_q[stage], kb * kBK, b_row, pol_w);
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
                    if (((filled >> s) & 1u) && !mbar_wait_short(&full_q[s], (fill_par >> s) & 1u))
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
                if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full_b[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_u32(sA + stage * kABytes);
                    const uint32_t b0 = smem_u32(sBb + stage * kBbBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32), IDESC,
                                    (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (++stage == kStages) {
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
            mma_commit(drain);
            if (!mbar_wait_short(drain, 0)) atomicOr(args.err, kErrTimeoutDrain);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ converters
        const int ct = threadIdx.x - 6 * 32;  // 0..255
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&full_q[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t* __restrict__ q = sBq + stage * kBqBytes;
                uint8_t* __restrict__ b = sBb + stage * kBbBytes;
                // BN rows x 4 items of 16 values; the two 8-value groups 2h, 2h+1 of row r go
                // to 16-byte units (2h) ^ (r % 8) and (2h+1) ^ (r % 8) of the row's 128 bytes
                // (the 128-byte swizzle the MMA reads).  All loads first, then the stores.
                constexpr int kItems = kBN * 4 / 256;  // per thread
                uint4 w[kItems];
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int i = ct + 256 * j;
                    w[j] = *reinterpret_cast<const uint4*>(q + (i >> 2) * kBK + (i & 3) * 16);
                }
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int i = ct + 256 * j;
                    const int r = i >> 2, h = i & 3;
                    uint8_t* row = b + r * 128;
                    *reinterpret_cast<uint4*>(row + (((2 * h) ^ (r & 7)) << 4)) = i8x8_to_bf16(make_uint2(w[j].x, w[j].y));
                    *reinterpret_cast<uint4*>(row + (((2 * h + 1) ^ (r & 7)) << 4)) =
                        i8x8_to_bf16(make_uint2(w[j].z, w[j].w));
                }
                fence_proxy_async_shared();  // generic-proxy writes -> tensor-core reads
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_b[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            if (lane == 0) atomicOr(args.err, kErrTimeoutProducer);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
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
            if (!mbar_wait(&tfull[acc], (it >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int row = m * kBM + r_in_tile;
            const bool row_ok = row < s_rows[tm.g];
            __nv_bfloat16* orow = out + (size_t)(s_roff[tm.g] + row) * args.ldo;
            const size_t cb = (size_t)tm.g * args.b_rows_per_group;
            epilogue_q8<ACT>(tmem_base + acc * kBN + (static_cast<uint32_t>(q * 32) << 16), orow, row_ok,
                             n * OUT_COLS, args.N, args.scale + cb, GATED ? args.scale3 + cb : nullptr,
                             bias != nullptr ? bias + cb : nullptr);
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

template <int ACT>
cudaError_t launch_t(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& q3, const GroupedGemmQ8Args& args,
                     int grid, cudaStream_t st, bool pdl)
{
    auto kern = k_grouped_gemm_q8<ACT>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), kSmem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), kSmem, st, pdl, a, q, q3, args);
}

// One warp per row: scale = max|w| / 127, q = rint(w / scale) (IEEE fp32 division).
template <typename T>
__global__ void __launch_bounds__(256) k_quantize_int8(const T* __restrict__ w, long long rows, int cols,
                                                       int8_t* __restrict__ q, float* __restrict__ scale)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long r = (long long)blockIdx.x * 8 + warp; r < rows; r += (long long)gridDim.x * 8) {
        const T* row = w + r * cols;
        float amax = 0.0f;
        for (int c = lane; c < cols; c += 32) amax = fmaxf(amax, fabsf(to_f32(row[c])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax / 127.0f;
        if (lane == 0) scale[r] = s;
        for (int c = lane; c < cols; c += 32) {
            float t = s > 0.0f ? rintf(to_f32(row[c]) / s) : 0.0f;
            t = fminf(fmaxf(t, -127.0f), 127.0f);
            q[r * cols + c] = (int8_t)t;
        }
    }
}

}  // namespace

size_t gemm_q8_smem() { return kSmem; }

cudaError_t launch_gemm_q8(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& q3,
                           const GroupedGemmQ8Args& args, int act, int grid, cudaStream_t st, bool pdl)
{
    switch (act) {
    case kActNone: return launch_t<kActNone>(a, q, q3, args, grid, st, pdl);
    case kActRelu: return launch_t<kActRelu>(a, q, q3, args, grid, st, pdl);
    case kActGeluTanh: return launch_t<kActGeluTanh>(a, q, q3, args, grid, st, pdl);
    case kActGeluErf: return launch_t<kActGeluErf>(a, q, q3, args, grid, st, pdl);
    default: return launch_t<kActSwiglu>(a, q, q3, args, grid, st, pdl);
    }
}

cudaError_t launch_quantize_int8(const void* w, bool bf16, long long rows, int cols, int8_t* q, float* scale,
                                 int sms, cudaStream_t st)
{
    long long grid = (rows + 7) / 8;
    if (grid > (long long)sms * 32) grid = (long long)sms * 32;
    if (grid < 1) grid = 1;
    if (bf16)
        return launch_kernel(k_quantize_int8<__nv_bfloat16>, dim3((int)grid), dim3(256), 0, st, false,
                             static_cast<const __nv_bfloat16*>(w), rows, cols, q, scale);
    return launch_kernel(k_quantize_int8<float>, dim3((int)grid), dim3(256), 0, st, false,
                         static_cast<const float*>(w), rows, cols, q, scale);
}

}  // namespace moe
