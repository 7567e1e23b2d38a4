// router_tc.cu -- stage 1 of bf16 layers on the tensor core: router logits.
//
// The router must run in fp32 ("MoE 混合专家模型串讲" §"选择性精度"), but the
// logits x W_gate^T are a dense contraction.  x is bf16 already, so it is
// exact; W_gate (fp32) is split exactly into three bf16 terms
//     W = W_hi + W_mid + W_lo,  W_hi = bf16(W), W_mid = bf16(W - W_hi),
//     W_lo = bf16(W - W_hi - W_mid)        (residual error <= 2^-24 |W|)
// (the split-precision bfloat16 method of Henry, Tang and Heinecke, "Leveraging
// the bfloat16 artificial intelligence datatype for higher-precision
// computations", 2019).  Every bf16 x bf16 product is exact in fp32.
//
// The tensor core adds each MMA's partial products into the TMEM accumulator
// with less than IEEE fp32 precision, so the error of one long accumulation
// chain grows with its length (3 d / 16 MMAs).  The K loop is therefore cut
// into chunks of a few K-blocks: each chunk accumulates in one of two TMEM
// accumulators (alternating, so the MMAs of chunk c+1 overlap the drain of
// chunk c), and the epilogue warps add every finished chunk into fp32
// registers with round-to-nearest additions.  The error is then bounded by the
// chunk length, independent of d, and comparable to an fp32 FFMA dot product.
//
// k_split_wgate writes the three terms in blocks of 16 experts,
// [E_pad / 16][3][16][d] bf16 (rows >= E zero, E_pad a multiple of 64): a tile of
// BN experts (16, 32 or 64) is BN / 16 consecutive blocks, so one TMA box of 3 BN
// rows holds its three terms whatever BN is, and the split depends on W_gate
// alone -- it can be made once per weight update (moe_prepare_router_weights) or
// by every call into the workspace.  k_router_logits_tc: persistent, one CTA per
// SM, warp-specialised like the grouped GEMM: warp 0 TMA (x tile 128 x 64 and one
// box of the tile's 3 BN term rows per stage), warp 1 tcgen05.mma (M = 128, N = 3 BN:
// the hi, mid and lo products of a K-step in one instruction; accumulator column
// 48 b + 16 q + j holds term q of expert 16 b + j of the tile), warps 2-5 epilogue
// (chunk promotion (lo + mid) + hi into fp32 registers, bias add, fp32 logits to
// global).  Softmax, top-k and gates follow in k_router_topk (router.cu).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRBM = 128;
constexpr int kRBK = 64;
constexpr int kRThreads = 192;
// K-blocks (of 64) per TMEM accumulation chunk: 2 for wide expert tiles; 4 for
// BN <= 32, where a chunk's MMAs are short and the per-chunk promotion would
// dominate (the error bound doubles and stays below the fp32 FFMA router's)
template <int BN>
constexpr int chunk_kb() { return BN <= 32 ? 4 : 2; }

// BN = experts per tile; the three split terms of the tile's experts are stacked
// along the MMA's N dimension (N = 3 BN): one MMA per K-step covers all three.
template <int BN>
struct RCfg {
    static constexpr int N = 3 * BN;
    static constexpr uint32_t A_BYTES = kRBM * kRBK * 2;
    static constexpr uint32_t B_BYTES = N * kRBK * 2;  // the three splits
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_FIT = 196608 / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr uint32_t TMEM_COLS = 2 * N <= 32 ? 32 : 2 * N <= 64 ? 64 : 2 * N <= 128 ? 128 : 2 * N <= 256 ? 256 : 512;
    static constexpr size_t SMEM = 1024 + STAGES * (size_t)STAGE_BYTES + 256;
};

// The three bf16 terms of one fp32 weight: hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid); both differences are exact in fp32.
__device__ __forceinline__ void split3(float w, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

// out is [E_pad / 16][3][16][d]: for each block of 16 experts, its hi, mid and lo rows
// (rows >= E zero).  With d a multiple of 8 and W_gate 16-byte aligned every thread
// splits 8 consecutive weights of a row (two 16-byte loads, three 16-byte stores);
// otherwise one weight.
constexpr int kSplitBlock = 16;
__global__ void __launch_bounds__(256) k_split_wgate(const float* __restrict__ Wg, int E, int E_pad, int d,
                                                     __nv_bfloat16* __restrict__ out)
{
    griddep_launch_dependents();
    griddep_wait();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    if ((d & 7) == 0 && (reinterpret_cast<uintptr_t>(Wg) & 15u) == 0) {
        const size_t n8 = (size_t)E_pad * d / 8;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
            const int e = (int)(i * 8 / d), col = (int)(i * 8 - (size_t)e * d);
            float w[8];
            if (e < E) {
                const float4 u0 = __ldg(reinterpret_cast<const float4*>(Wg + (size_t)e * d + col));
                const float4 u1 = __ldg(reinterpret_cast<const float4*>(Wg + (size_t)e * d + col + 4));
                w[0] = u0.x, w[1] = u0.y, w[2] = u0.z, w[3] = u0.w;
                w[4] = u1.x, w[5] = u1.y, w[6] = u1.z, w[7] = u1.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q] = 0.0f;
            }
            __align__(16) __nv_bfloat16 h[8], m[8], lo[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) split3(w[q], h[q], m[q], lo[q]);
            const int blk = e / kSplitBlock, el = e - blk * kSplitBlock;
            const size_t r0 = (size_t)blk * 3 * kSplitBlock + el;  // hi row; mid and lo rows 16 and 32 further
            *reinterpret_cast<uint4*>(out + r0 * d + col) = *reinterpret_cast<const uint4*>(h);
            *reinterpret_cast<uint4*>(out + (r0 + kSplitBlock) * d + col) = *reinterpret_cast<const uint4*>(m);
            *reinterpret_cast<uint4*>(out + (r0 + 2 * kSplitBlock) * d + col) = *reinterpret_cast<const uint4*>(lo);
        }
        return;
    }
    const size_t n = (size_t)E_pad * d;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int e = (int)(i / d), col = (int)(i - (size_t)e * d);
        const float w = e < E ? Wg[i] : 0.0f;  // Wg is [E, d]: the same flat index for e < E
        __nv_bfloat16 h, m, lo;
        split3(w, h, m, lo);
        const int blk = e / kSplitBlock, el = e - blk * kSplitBlock;
        const size_t r0 = (size_t)blk * 3 * kSplitBlock + el;
        out[r0 * d + col] = h;
        out[(r0 + kSplitBlock) * d + col] = m;
        out[(r0 + 2 * kSplitBlock) * d + col] = lo;
    }
}

__device__ __forceinline__ bool wait_short(uint64_t* bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 100000000ull) return false;  // 100 ms
    return true;
}


// The rest of the router for one token per thread when a tile holds every expert:
// logits (+ bias) written out, softmax, the k largest logits (ties to the lower expert
// index, a NaN logit competing as -inf), gates (renormalised over the k when asked),
// probabilities if asked, and the column sums of p over the warp's 32 tokens (one
// psum_part row per 32-token group, router_blocks(T) rows in all).  Every lane of
// the warp must call it (the column sums are warp reductions); rows >= T add nothing.
template <int BN>
__device__ __forceinline__ void route_rows(const float (&sum)[BN], int row, int group, const RouterGemmArgs& a)
{
    const bool valid = row < a.T;
    const int E = a.E;
    float l[BN];
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < BN; ++e) {
        l[e] = e < E ? sum[e] + (a.bg != nullptr ? a.bg[e] : 0.0f) : -INFINITY;
        mx = fmaxf(mx, l[e]);
    }
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < BN; ++e) s += e < E ? expf(l[e] - mx) : 0.0f;
    const float inv = 1.0f / s;
    if (valid) {
        float* lrow = a.logits + (size_t)row * E;
#pragma unroll
        for (int e = 0; e < BN; ++e)
            if (e < E) lrow[e] = l[e];
        // top-k rounds over (logit desc, expert asc)
        uint64_t taken = 0;
        float gsum = 0.0f;
        for (int r = 0; r < a.k; ++r) {
            float bv = -INFINITY;
            int be = -1;
#pragma unroll
            for (int e = 0; e < BN; ++e) {
                const float v = (l[e] != l[e]) ? -INFINITY : l[e];
                if (e < E && !((taken >> e) & 1ull) && (be < 0 || v > bv)) {
                    bv = v;
                    be = e;
                }
            }
            taken |= 1ull << be;
            float le = 0.0f;
#pragma unroll
            for (int e = 0; e < BN; ++e)
                if (e == be) le = l[e];
            const float pe = expf(le - mx) * inv;
            a.idx[(size_t)row * a.k + r] = be;
            a.gates[(size_t)row * a.k + r] = pe;
            gsum += pe;
        }
        if (a.renormalize)
            for (int r = 0; r < a.k; ++r) a.gates[(size_t)row * a.k + r] /= gsum;
    }
    // probabilities and their column sums over the warp's rows
    const int lane = threadIdx.x & 31;
    float mine = 0.0f;  // lane e ends with expert e's sum (lanes 0..31), the rest in a loop
#pragma unroll
    for (int e = 0; e < BN; ++e) {
        float pe = (valid && e < E) ? expf(l[e] - mx) * inv : 0.0f;
        if (valid && e < E && a.probs != nullptr) a.probs[(size_t)row * E + e] = pe;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pe += __shfl_xor_sync(0xffffffffu, pe, o);
        if ((e & 31) == lane) mine = pe;
        if ((e & 31) == 31 || e == BN - 1) {  // a batch of 32 experts is complete
            const int e0 = e & ~31;
            if (group * 32 < a.T && e0 + lane < E && e0 + lane <= e) a.psum_part[(size_t)group * E + e0 + lane] = mine;
        }
    }
}

template <int BN, bool FUSE>
__global__ void __launch_bounds__(kRThreads, 1)
    k_router_logits_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const RouterGemmArgs a)
{
    using C = RCfg<BN>;
    constexpr uint32_t IDESC = idesc_bf16_f32(kRBM, C::N);

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

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&tfull[q], 1);
            mbar_init(&tempty[q], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();  // x and the W_gate splits may come from earlier kernels
    if (FUSE && blockIdx.x == 0 && threadIdx.x == 0) *a.scan_done = 0u;  // re-arm the dispatch scan

    const int m_tiles = ceil_div(a.T, kRBM);
    const int total = m_tiles * a.n_tiles * a.k_splits;
    const int num_kb_all = ceil_div(a.d, kRBK);
    const int kb_per_split = ceil_div(num_kb_all, a.k_splits);

    if (warp == 0) {
        if (lane == 0) {
            // W is re-read by every M-tile and x by every expert tile; with one expert
            // tile x streams through once and is marked evict-first
            const uint64_t pol = policy_evict_last();
            const uint64_t pol_x = a.n_tiles > 1 ? pol : policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int mn = tile % (m_tiles * a.n_tiles), ks = tile / (m_tiles * a.n_tiles);
                const int m = mn / a.n_tiles, n = mn - m * a.n_tiles;
                const int kbeg = ks * kb_per_split;
                const int kend = min(kbeg + kb_per_split, num_kb_all);
                for (int kb = kbeg; kb < kend; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d(sA + stage * C::A_BYTES, &tmX, &full[stage], kb * kRBK, m * kRBM, pol_x);
                    tma_load_2d(sB + stage * C::B_BYTES, &tmW, &full[stage], kb * kRBK, n * C::N, pol);
                    filled |= 1u << stage;
                    fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(a.err, kErrTimeoutProducer);
                *abort_flag = 1;
                for (int s = 0; s < C::STAGES; ++s)
                    if (((filled >> s) & 1u) && !wait_short(&full[s], (fill_par >> s) & 1u))
                        atomicOr(a.err, kErrTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, ci = 0;  // ci counts accumulation chunks over all tiles of this CTA
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int ks = tile / (m_tiles * a.n_tiles);
                const int kbeg = ks * kb_per_split;
                const int num_kb = min(kbeg + kb_per_split, num_kb_all);
                for (int kb0 = kbeg; kb0 < num_kb && ok; kb0 += chunk_kb<BN>(), ++ci) {
                    const int acc = ci & 1;
                    if (!mbar_wait(&tempty[acc], ((ci >> 1) & 1) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + acc * C::N;
                    const int kb1 = kb0 + chunk_kb<BN>() < num_kb ? kb0 + chunk_kb<BN>() : num_kb;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full[stage], phase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
                        const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
                        // hi, mid and lo terms land in column groups [0, BN), [BN, 2 BN), [2 BN, 3 BN)
#pragma unroll
                        for (int k = 0; k < kRBK / 16; ++k)
                            mma_bf16_ss(d_tmem, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32),
                                        IDESC, (kb == kb0 && k == 0) ? 0u : 1u);
                        mma_commit(&empty[stage]);
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&tfull[acc]);
                }
            }
            if (!ok) {
                atomicOr(a.err, kErrTimeoutMma);
                *abort_flag = 1;
            }
            mma_commit(drain);
            if (!wait_short(drain, 0)) atomicOr(a.err, kErrTimeoutDrain);
        }
    } else {
        const int q = warp & 3;
        bool ok = true;
        int ci = 0;
        const bool vec = (a.E % 4) == 0;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const int mn = tile % (m_tiles * a.n_tiles), ks = tile / (m_tiles * a.n_tiles);
            const int m = mn / a.n_tiles, n = mn - m * a.n_tiles;
            const int kbeg = ks * kb_per_split;
            const int num_kb = min(kbeg + kb_per_split, num_kb_all);
            float sum[BN];
#pragma unroll
            for (int i = 0; i < BN; ++i) sum[i] = 0.0f;
            for (int kb0 = kbeg; kb0 < num_kb; kb0 += chunk_kb<BN>(), ++ci) {
                const int acc = ci & 1;
                if (!mbar_wait(&tfull[acc], (ci >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t t_lane = tmem_base + acc * C::N + (static_cast<uint32_t>(q * 32) << 16);
                // promote the chunk: (lo + mid) + hi per expert, added to the fp32 running
                // sums; block b of 16 experts has its hi, mid, lo columns at 48 b + {0, 16, 32}
#pragma unroll
                for (int c = 0; c < BN / kSplitBlock; ++c) {
                    uint32_t rh[16], rm[16], rl[16];
                    tmem_ld_16cols(t_lane + c * 3 * kSplitBlock, rh);
                    tmem_ld_16cols(t_lane + c * 3 * kSplitBlock + kSplitBlock, rm);
                    tmem_ld_16cols(t_lane + c * 3 * kSplitBlock + 2 * kSplitBlock, rl);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        sum[c * 16 + i] += (__uint_as_float(rl[i]) + __uint_as_float(rm[i])) + __uint_as_float(rh[i]);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
            }
            if (!ok) break;
            const int row = m * kRBM + q * 32 + lane;
            if constexpr (FUSE) {
                route_rows<BN>(sum, row, m * 4 + q, a);
                continue;
            }
            if (row < a.T) {
                // one K range: partial sums without bias, summed by the top-k kernel
                const bool split = a.k_splits > 1;
                float* lrow = a.logits + ((size_t)ks * a.T + row) * a.E;
#pragma unroll
                for (int i = 0; i < BN; i += 4) {
                    const int col = n * BN + i;
                    float o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        o[u] = sum[i + u] + ((!split && a.bg != nullptr && col + u < a.E) ? a.bg[col + u] : 0.0f);
                    if (vec && col + 4 <= a.E) {
                        *reinterpret_cast<float4*>(lrow + col) = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (col + u < a.E) lrow[col + u] = o[u];
                    }
                }
            }
        }
        if (!ok) {
            if (lane == 0) atomicOr(a.err, kErrTimeoutEpilogue);
            *abort_flag = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int BN, bool FUSE>
cudaError_t launch_bn(const CUtensorMap& x, const CUtensorMap& w, const RouterGemmArgs& a, int sms,
                      cudaStream_t st, bool pdl)
{
    auto kern = k_router_logits_tc<BN, FUSE>;
    const size_t smem = RCfg<BN>::SMEM;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int tiles = ceil_div(a.T, kRBM) * a.n_tiles * a.k_splits;
    return launch_kernel(kern, dim3(tiles < sms ? tiles : sms), dim3(kRThreads), smem, st, pdl, x, w, a);
}

}  // namespace

int router_tc_bn(int T, int E)
{
    // Aim for about 128 CTAs (m-tiles x expert tiles), BN a power of two in [16, 128].
    const int m_tiles = T > 0 ? ceil_div(T, kRBM) : 1;
    const int want_tiles = ceil_div(128, m_tiles);
    const int per_tile = ceil_div(E, want_tiles);
    int bn = 16;
    while (bn < per_tile && bn < 64) bn *= 2;  // 3 bn <= 256 columns per MMA
    return bn;
}

int router_tc_ksplits(int T, int E, int d)
{
    // split K only when the (M-tile, expert-tile) grid is far below ~128 CTAs, keeping
    // at least 8 K-blocks per split
    const int tiles = ceil_div(T, kRBM) * ceil_div(E, router_tc_bn(T, E));
    int ks = 1;
    while (ks < 8 && tiles * ks * 2 <= 128 && ceil_div(d, kRBK) >= 16 * ks) ks *= 2;
    return ks;
}

int router_split_rows(int E) { return (E + 63) / 64 * 64; }

cudaError_t launch_split_wgate(const float* Wg, int E, int d, void* out, int sms, cudaStream_t st, bool pdl)
{
    const int E_pad = router_split_rows(E);
    const size_t n = (d % 8 == 0) ? (size_t)E_pad * d / 8 : (size_t)E_pad * d;
    size_t grid = (n + 255) / 256;
    if (grid > (size_t)sms * 8) grid = (size_t)sms * 8;
    return launch_kernel(k_split_wgate, dim3((int)grid), dim3(256), 0, st, pdl, Wg, E, E_pad, d,
                         static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_router_logits_tc(const CUtensorMap& x, const CUtensorMap& w, const RouterGemmArgs& a,
                                    int bn, int sms, cudaStream_t st, bool pdl)
{
    // a.fuse is set only for tiles of at most 32 experts (one tile, no K split): there the
    // epilogue's per-token softmax and top-k are short; wider tiles keep the top-k kernel
    switch (bn) {
    case 16: return a.fuse ? launch_bn<16, true>(x, w, a, sms, st, pdl) : launch_bn<16, false>(x, w, a, sms, st, pdl);
    case 32: return a.fuse ? launch_bn<32, true>(x, w, a, sms, st, pdl) : launch_bn<32, false>(x, w, a, sms, st, pdl);
    default: return launch_bn<64, false>(x, w, a, sms, st, pdl);
    }
}

}  // namespace moe
