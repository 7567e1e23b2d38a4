// router.cu -- stage 1 of the layer: the fp32 softmax router and top-k.
//
// logits[t,e] = sum_i x[t,i] * W_gate[e,i] (+ b_gate[e]), accumulated in fp32
// ("混合专家 MOE 是什么" §"公式：三步走": g = softmax(W_g x); the router is
// computed in fp32 as "MoE 混合专家模型串讲" §"选择性精度" prescribes).
// p = softmax over the E routed experts; the k largest logits are selected
// with warp reductions (redux.sync max/min), ties to the lower expert index ("混合专家模型MoE
// 入门实战" §3.3 torch.topk; "MoE架构解析" §2.1 top_k on the logits - the same
// experts, softmax being monotone).  Gates are p, or p divided by the sum of
// the k selected p ("混合专家模型MoE入门实战" §3.3 重新归一化).
//
// One block = 32 tokens = 8 warps x 4 tokens; lane l of a warp owns experts
// l, l+32, ... (EJ of them), so after the d-loop every warp holds full logit
// rows of its tokens in registers and finishes softmax/top-k with warp reductions.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouterBK = 16;  // d-chunk staged in shared memory
constexpr int kTokPerWarp = kRouterTokens / 8;

// Order-preserving 32-bit key of a logit for the top-k: a larger float gets a larger
// key, NaN competes as -inf and -0 as +0 (so equal logits tie and the lower expert
// index wins).  Every key of a real candidate is >= key(-inf) = 0x007fffff > 0, so 0
// marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float v)
{
    v = (v != v) ? -INFINITY : (v == 0.0f ? 0.0f : v);
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Softmax, top-k and gates of one token from its logit row l (lane owns experts
// lane, lane+32, ...; -inf beyond E), executed by a whole warp.  Adds the token's
// probabilities to the lane's running column sums.  write_logits = false when
// the logits row already sits in a.logits.
template <int EJ>
__device__ __forceinline__ void route_token(const float (&l)[EJ], int t, const RouterArgs& a,
                                            bool write_logits, float (&psum)[EJ])
{
    const int lane = threadIdx.x & 31;
    uint32_t key[EJ];
    uint32_t kmax = 0;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
        key[j] = (lane + 32 * j < a.E) ? order_key(l[j]) : 0u;
        kmax = max(kmax, key[j]);
    }
    // the row maximum (NaN ignored) by one warp reduction of the keys
    const float m = key_value(__reduce_max_sync(0xffffffffu, kmax));
    float p[EJ];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        p[j] = (e < a.E) ? expf(l[j] - m) : 0.0f;
        s += p[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        p[j] *= inv;
        psum[j] += p[j];
        if (e < a.E) {
            if (write_logits && a.logits) a.logits[(size_t)t * a.E + e] = l[j];
            if (a.probs) a.probs[(size_t)t * a.E + e] = p[j];
        }
    }

    // top-k: k rounds of a warp argmax over (logit desc, expert asc), each two warp
    // reductions: the largest key among the lanes' best untaken candidates, then the
    // lowest expert holding it.  A lane's best is its first (lowest-index) maximum, so
    // the lowest expert with the round's key is the lowest of those lanes' bests.
    // k <= E, so every round finds an expert.
    int my_e = 0;
    float my_p = 0.0f, gsum = 0.0f;
    for (int r = 0; r < a.k; ++r) {
        uint32_t lk = 0u, le = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < EJ; ++j)
            if (key[j] > lk) {
                lk = key[j];
                le = (uint32_t)(lane + 32 * j);
            }
        const uint32_t rk = __reduce_max_sync(0xffffffffu, lk);
        const int be = (int)__reduce_min_sync(0xffffffffu, lk == rk ? le : 0xffffffffu);
        const int bj = be >> 5;
        float pj = 0.0f;
#pragma unroll
        for (int j = 0; j < EJ; ++j)
            if (j == bj) pj = p[j];
        const float bp = __shfl_sync(0xffffffffu, pj, be & 31);
        if ((be & 31) == lane) {
#pragma unroll
            for (int j = 0; j < EJ; ++j)
                if (j == bj) key[j] = 0u;  // taken
        }
        if (lane == r) {
            my_e = be;
            my_p = bp;
        }
        gsum += bp;
    }
    if (lane < a.k) {
        a.idx[(size_t)t * a.k + lane] = my_e;
        a.gates[(size_t)t * a.k + lane] = a.renormalize ? my_p / gsum : my_p;
    }
}

// Deterministic per-block column sums of p (warps in order, each warp's tokens in
// order) into a.psum_part[blockIdx.x].  `scratch` holds WARPS x 32*EJ floats.
template <int EJ, int WARPS = 8>
__device__ __forceinline__ void block_psum(const float (&psum)[EJ], float* scratch, const RouterArgs& a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < EJ; ++j) scratch[warp * 32 * EJ + lane + 32 * j] = psum[j];
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += WARPS * 32) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s += scratch[w * 32 * EJ + e];
        a.psum_part[(size_t)blockIdx.x * a.E + e] = s;
    }
}

template <typename TX, int EJ>
__global__ void __launch_bounds__(256) k_router(RouterArgs a)
{
    constexpr int kWsStride = kRouterBK + 1;  // conflict-free column reads
    __shared__ float xs[kRouterTokens][kRouterBK];
    __shared__ float ws[32 * EJ * kWsStride];  // reused for the column sums afterwards

    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRouterTokens;
    const TX* x = static_cast<const TX*>(a.x);

    if (blockIdx.x == 0 && threadIdx.x == 0) *a.scan_done = 0u;  // re-arm the dispatch scan

    float acc[kTokPerWarp][EJ];
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < a.d; k0 += kRouterBK) {
        // x tile: 32 tokens x 16 columns, one element per thread pair
        for (int v = threadIdx.x; v < kRouterTokens * kRouterBK; v += 256) {
            const int r = v / kRouterBK, c = v % kRouterBK;
            const int t = t0 + r, col = k0 + c;
            xs[r][c] = (t < a.T && col < a.d) ? to_f32(x[(size_t)t * a.d + col]) : 0.0f;
        }
        for (int v = threadIdx.x; v < 32 * EJ * kRouterBK; v += 256) {
            const int r = v / kRouterBK, c = v % kRouterBK;
            const int col = k0 + c;
            ws[r * kWsStride + c] = (r < a.E && col < a.d) ? a.Wg[(size_t)r * a.d + col] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kRouterBK; ++kk) {
            float xv[kTokPerWarp];
#pragma unroll
            for (int i = 0; i < kTokPerWarp; ++i) xv[i] = xs[warp * kTokPerWarp + i][kk];
#pragma unroll
            for (int j = 0; j < EJ; ++j) {
                const float wv = ws[(lane + 32 * j) * kWsStride + kk];
#pragma unroll
                for (int i = 0; i < kTokPerWarp; ++i) acc[i][j] = fmaf(xv[i], wv, acc[i][j]);
            }
        }
        __syncthreads();
    }

    if (a.raw_out != nullptr) {  // projection only (the noise logits of noisy gating)
#pragma unroll
        for (int i = 0; i < kTokPerWarp; ++i) {
            const int t = t0 + warp * kTokPerWarp + i;
            if (t >= a.T) break;
#pragma unroll
            for (int j = 0; j < EJ; ++j) {
                const int e = lane + 32 * j;
                if (e < a.E) a.raw_out[(size_t)t * a.E + e] = acc[i][j];
            }
        }
        return;
    }

    float bias[EJ], nbias[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        bias[j] = (a.bg != nullptr && e < a.E) ? a.bg[e] : 0.0f;
        nbias[j] = (a.bn != nullptr && e < a.E) ? a.bn[e] : 0.0f;
    }

    float psum[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) psum[j] = 0.0f;

#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i) {
        const int t = t0 + warp * kTokPerWarp + i;
        if (t >= a.T) break;  // warp-uniform
        float l[EJ];
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            const int e = lane + 32 * j;
            l[j] = (e < a.E) ? acc[i][j] + bias[j] : -INFINITY;
            if (a.eps != nullptr && e < a.E) {
                const size_t o = (size_t)t * a.E + e;
                l[j] += a.eps[o] * (softplus_f32(a.noise_parts[o] + nbias[j]) + a.min_std);
            }
        }
        route_token<EJ>(l, t, a, true, psum);
    }

    // the d-loop ended with a barrier: the weight tile is free for the column sums
    block_psum<EJ>(psum, ws, a);
}

// Softmax / top-k / gates for logits already in a.logits (computed by the
// tensor-core router GEMM), or for the sum of split-K partial logits plus the bias.
// NOISY: the noise of noisy top-k gating is added first ("MoE架构解析" §2.1
// noisy_top_k_gating; "MoE 混合专家模型串讲" §"代码实战" NoisyTop1Gate), so softmax,
// top-k, gates and the column sums all see the noisy logits, which are written out.
// A block covers kTopkTokens tokens, one per warp, and writes one row of column
// sums of p (router_topk_blocks(T) rows in all): a small batch still spreads over
// many SMs.
template <int EJ, int WARPS, bool NOISY>
__global__ void __launch_bounds__(WARPS * 32) k_router_topk(RouterArgs a)
{
    constexpr int TPW = kTopkTokens / WARPS;  // tokens per warp
    __shared__ float scratch[WARPS * 32 * EJ];
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kTopkTokens;
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.scan_done = 0u;  // re-arm the dispatch scan
    float psum[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) psum[j] = 0.0f;
    // all loads of the warp's tokens first, then the dependent reduction chains
    float l[TPW][EJ];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            const int t = t0 + warp * TPW + i, e = lane + 32 * j;
            const bool in = t < a.T && e < a.E;
            l[i][j] = in ? (a.logit_parts == nullptr ? a.logits[(size_t)t * a.E + e] : 0.0f) : -INFINITY;
        }
    if (a.logit_parts != nullptr) {
        // split-K: add the partial sums in K order; the loads of PF splits are issued
        // before their additions
        constexpr int PF = TPW * EJ <= 8 ? 8 : TPW * EJ <= 16 ? 4 : 1;
        for (int ks0 = 0; ks0 < a.k_splits; ks0 += PF) {
            float v[PF][TPW][EJ];
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                const float* part = a.logit_parts + (size_t)(ks0 + u) * a.T * a.E;
#pragma unroll
                for (int i = 0; i < TPW; ++i)
#pragma unroll
                    for (int j = 0; j < EJ; ++j) {
                        const int t = t0 + warp * TPW + i, e = lane + 32 * j;
                        v[u][i][j] = (ks0 + u < a.k_splits && t < a.T && e < a.E) ? __ldcg(&part[(size_t)t * a.E + e])
                                                                                  : 0.0f;
                    }
            }
#pragma unroll
            for (int u = 0; u < PF; ++u)
#pragma unroll
                for (int i = 0; i < TPW; ++i)
#pragma unroll
                    for (int j = 0; j < EJ; ++j)
                        if (ks0 + u < a.k_splits) l[i][j] += v[u][i][j];
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int j = 0; j < EJ; ++j) {
                const int e = lane + 32 * j;
                if (a.bg != nullptr && e < a.E) l[i][j] += a.bg[e];
            }
    }
    if constexpr (NOISY) {
        // noise logits: split-K partials in K order, then the bias; then the noisy logits
        float nz[TPW][EJ];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int j = 0; j < EJ; ++j) nz[i][j] = 0.0f;
        for (int ks = 0; ks < a.k_splits; ++ks) {
            const float* part = a.noise_parts + (size_t)ks * a.T * a.E;
#pragma unroll
            for (int i = 0; i < TPW; ++i)
#pragma unroll
                for (int j = 0; j < EJ; ++j) {
                    const int t = t0 + warp * TPW + i, e = lane + 32 * j;
                    if (t < a.T && e < a.E) nz[i][j] += part[(size_t)t * a.E + e];
                }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int j = 0; j < EJ; ++j) {
                const int t = t0 + warp * TPW + i, e = lane + 32 * j;
                if (t < a.T && e < a.E) {
                    const float z = nz[i][j] + (a.bn != nullptr ? a.bn[e] : 0.0f);
                    l[i][j] += a.eps[(size_t)t * a.E + e] * (softplus_f32(z) + a.min_std);
                }
            }
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = t0 + warp * TPW + i;
        if (t >= a.T) break;  // warp-uniform
        route_token<EJ>(l[i], t, a, NOISY || a.logit_parts != nullptr, psum);
    }
    block_psum<EJ, WARPS>(psum, scratch, a);
}

template <typename TX>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t st, bool pdl)
{
    const dim3 grid(ceil_div(a.T, kRouterTokens)), block(256);
    if (a.E <= 32) return launch_kernel(k_router<TX, 1>, grid, block, 0, st, pdl, a);
    if (a.E <= 64) return launch_kernel(k_router<TX, 2>, grid, block, 0, st, pdl, a);
    if (a.E <= 128) return launch_kernel(k_router<TX, 4>, grid, block, 0, st, pdl, a);
    if (a.E <= 256) return launch_kernel(k_router<TX, 8>, grid, block, 0, st, pdl, a);
    return launch_kernel(k_router<TX, 16>, grid, block, 0, st, pdl, a);
}

template <int EJ>
cudaError_t launch_topk_ej(const RouterArgs& a, cudaStream_t st)
{
    constexpr int WARPS = kTopkTokens;
    const dim3 grid(router_topk_blocks(a.T)), block(WARPS * 32);
    if (a.eps != nullptr) return launch_kernel(k_router_topk<EJ, WARPS, true>, grid, block, 0, st, true, a);
    return launch_kernel(k_router_topk<EJ, WARPS, false>, grid, block, 0, st, true, a);
}

}  // namespace

int router_blocks(int T) { return ceil_div(T, kRouterTokens); }

int router_topk_blocks(int T) { return ceil_div(T, kTopkTokens); }

cudaError_t launch_router_topk(const RouterArgs& a, cudaStream_t st)
{
    if (a.E <= 32) return launch_topk_ej<1>(a, st);
    if (a.E <= 64) return launch_topk_ej<2>(a, st);
    if (a.E <= 128) return launch_topk_ej<4>(a, st);
    if (a.E <= 256) return launch_topk_ej<8>(a, st);
    return launch_topk_ej<16>(a, st);
}

cudaError_t launch_router(const RouterArgs& a, bool bf16, cudaStream_t st, bool pdl)
{
    return bf16 ? launch_router_t<__nv_bfloat16>(a, st, pdl) : launch_router_t<float>(a, st, pdl);
}

}  // namespace moe
