// backward.cu -- the memory-bound kernels of the layer's backward pass.
//
// The backward of y[t] = sum_j g[t,j] e_j(x[t]) + shared(x[t]) + pass(t) x[t]
// ("混合专家模型MoE入门实战" §3.4-§3.5: the layer is trained end to end with
// task loss + coef * aux loss):
//   k_bwd_combine    dYp[row(t,j)] = g[t,j] dy[t];  dg[t,j] = <dy[t], Yp[row(t,j)]>
//   k_router_bwd     dp from dg (through the renormalisation when it applies) and
//                    from the balance statistic (P_i differentiable, f_i not:
//                    "MoE 混合专家模型串讲" §"负载均衡损失函数"), then the softmax
//                    Jacobian dl = p (dp - <p, dp>); under noisy gating also
//                    dn = dl eps sigmoid(n) for the noise projection
//   k_colsum         bias gradients: column sums over the rows of each segment
//   k_bwd_unpermute  dx[t] = pass(t) dy[t] + sum_j dXp[row(t,j)] + dXs[t] + dx_router[t]
// The discrete choices of the forward (top-k, capacity drops) are held fixed.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p, size_t i) { return to_f32(p[i]); }

template <typename T>
__device__ __forceinline__ void st_round(T* p, size_t i, float v)
{
    if constexpr (sizeof(T) == 2) p[i] = __float2bfloat16_rn(v);
    else p[i] = v;
}

// One warp per token; 16-byte vectors of the row per lane.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_combine(BwdCombineArgs a)
{
    constexpr int V = Vec<T>::N;
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = a.d / V;
    const size_t row_bytes = (size_t)a.d * sizeof(T);
    for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
        const char* dyr = static_cast<const char*>(a.dy) + (size_t)t * row_bytes;
        for (int j = 0; j < a.k; ++j) {
            const size_t s = (size_t)t * a.k + j;
            const int r = a.slot_row[s];
            float dot = 0.0f;
            if (r >= 0) {
                const float g = a.gates[s];
                const char* yr = static_cast<const char*>(a.yp) + (size_t)r * row_bytes;
                char* dr = static_cast<char*>(a.dyp) + (size_t)r * row_bytes;
                for (int v = lane; v < nvec; v += 32) {
                    float u[V], y[V];
                    Vec<T>::load(dyr + v * 16, u);
                    Vec<T>::load(yr + v * 16, y);
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        dot = fmaf(u[i], y[i], dot);
                        u[i] *= g;
                    }
                    Vec<T>::store(dr + v * 16, u);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            }
            if (lane == 0) a.dgate[s] = dot;  // a dropped slot contributes nothing: 0
        }
    }
}

// One warp per token; lane l owns experts l, l + 32, ... (EJ of them).
template <int EJ>
__global__ void __launch_bounds__(256) k_router_bwd(RouterBwdArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float aux_scale = a.d_aux * (float)a.E / ((float)a.T * (float)a.T * (float)a.k);
    for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
        float l[EJ], p[EJ], dp[EJ];
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            const int e = lane + 32 * j;
            l[j] = e < a.E ? a.logits[(size_t)t * a.E + e] : -INFINITY;
            m = fmaxf(m, l[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            p[j] = (lane + 32 * j) < a.E ? expf(l[j] - m) : 0.0f;
            s += p[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float inv = 1.0f / s;
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            const int e = lane + 32 * j;
            p[j] *= inv;
            // balance statistic E * sum_e f_e P_e: d/dp[t,e] = E f_e / T, f_e = counts_e / (T k)
            dp[j] = e < a.E ? aux_scale * (float)a.counts[e] : 0.0f;
        }
        // the selected probabilities, sum and <dg, p_sel>
        float sel = 0.0f, dot = 0.0f;
        for (int jj = 0; jj < a.k; ++jj) {
            const size_t sl = (size_t)t * a.k + jj;
            const int e = a.idx[sl];
            float pe = 0.0f;
#pragma unroll
            for (int j = 0; j < EJ; ++j)
                if (j == (e >> 5)) pe = p[j];
            pe = __shfl_sync(0xffffffffu, pe, e & 31);
            sel += pe;
            dot += a.dgate[sl] * pe;
        }
        for (int jj = 0; jj < a.k; ++jj) {
            const size_t sl = (size_t)t * a.k + jj;
            const int e = a.idx[sl];
            const float dg = a.dgate[sl];
            const float add = a.renormalize ? dg / sel - dot / (sel * sel) : dg;
            if ((e & 31) == lane) {
#pragma unroll
                for (int j = 0; j < EJ; ++j)
                    if (j == (e >> 5)) dp[j] += add;
            }
        }
        float pdp = 0.0f;
#pragma unroll
        for (int j = 0; j < EJ; ++j) pdp = fmaf(p[j], dp[j], pdp);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pdp += __shfl_xor_sync(0xffffffffu, pdp, o);
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
            const int e = lane + 32 * j;
            if (e >= a.E) continue;
            const float g = p[j] * (dp[j] - pdp);
            const size_t o = (size_t)t * a.E + e;
            a.dl[o] = g;
            if (a.eps != nullptr) {
                float n = a.bn != nullptr ? a.bn[e] : 0.0f;
                for (int ks = 0; ks < a.k_splits; ++ks) n += a.noise_parts[(size_t)ks * a.T * a.E + o];
                a.dn[o] = g * a.eps[o] / (1.0f + expf(-n));
            }
        }
    }
}

// out[g][n] = sum over the rows of segment g of A[row][n].  A block covers (g, 32
// columns): lane = column, the 8 warps take every 8th row, then the 8 partial sums
// are added in warp order (deterministic).
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) k_colsum(ColsumArgs a)
{
    __shared__ float part[8][33];
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TI* A = static_cast<const TI*>(a.A);
    TO* out = static_cast<TO*>(a.out);
    const int chunks = ceil_div(a.N, 32);
    for (int item = blockIdx.x; item < a.G * chunks; item += gridDim.x) {
        const int g = item / chunks, n = (item - g * chunks) * 32 + lane;
        const long long r0 = a.row_off != nullptr ? a.row_off[g] : 0;
        const int rows = a.rows != nullptr ? a.rows[g] : a.fixed_rows;
        float s = 0.0f;
        if (n < a.N)
            for (int r = warp; r < rows; r += 8) s += to_f32(A[(r0 + r) * a.lda + n]);
        part[warp][lane] = s;
        __syncthreads();
        if (warp == 0 && n < a.N) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) t += part[w][lane];
            st_round(out, (size_t)(a.out_g0 + g) * a.N + n, t);
        }
        __syncthreads();
    }
}

// One warp per token, 16-byte vectors per lane, fp32 accumulation in a fixed order.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_unpermute(BwdUnpermuteArgs a)
{
    constexpr int V = Vec<T>::N;
    __shared__ int s_row[8][kMaxTopK];
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = a.d / V;
    const size_t row_bytes = (size_t)a.d * sizeof(T);
    for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
        const int r = lane < a.k ? a.slot_row[(size_t)t * a.k + lane] : -1;
        if (lane < a.k) s_row[warp][lane] = r;
        const unsigned dropped = __ballot_sync(0xffffffffu, lane < a.k && r < 0);
        const unsigned all_k = a.k >= 32 ? 0xffffffffu : ((1u << a.k) - 1u);
        const bool pass = a.residual_mode == 1 || dropped == all_k;
        __syncwarp();  // s_row visible to the whole warp
        const char* dyr = static_cast<const char*>(a.dy) + (size_t)t * row_bytes;
        const char* dxsr = a.dxs ? static_cast<const char*>(a.dxs) + (size_t)t * row_bytes : nullptr;
        const float* dxrr = a.dxr + (size_t)t * a.d;
        char* dxo = static_cast<char*>(a.dx) + (size_t)t * row_bytes;
        for (int v = lane; v < nvec; v += 32) {
            float acc[V];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = dxrr[v * V + i];
            if (pass) {
                float u[V];
                Vec<T>::load(dyr + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += u[i];
            }
            for (int j = 0; j < a.k; ++j) {
                const int rj = s_row[warp][j];
                if (rj < 0) continue;
                float u[V];
                Vec<T>::load(static_cast<const char*>(a.dxp) + (size_t)rj * row_bytes + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += u[i];
            }
            if (dxsr) {
                float u[V];
                Vec<T>::load(dxsr + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += u[i];
            }
            Vec<T>::store(dxo + v * 16, acc);
        }
        __syncwarp();  // s_row is rewritten for the warp's next token
    }
}

// One warp per (segment, pad row below the next 64-row boundary); 16-byte stores.
__global__ void __launch_bounds__(256) k_zero_pad_rows(ZeroPadArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int items = a.G * 64;
    for (int it = blockIdx.x * 8 + warp; it < items; it += gridDim.x * 8) {
        const int g = it >> 6, p = it & 63;
        const int kept = a.rows[g];
        const int end = (kept + 63) / 64 * 64;
        if (kept + p >= end) continue;
        const long long row = (long long)a.row_off[g] + kept + p;
        for (int b = 0; b < 3; ++b) {
            if (a.buf[b] == nullptr) continue;
            uint4* r = reinterpret_cast<uint4*>(static_cast<char*>(a.buf[b]) + row * a.row_bytes[b]);
            for (int v = lane; v < a.row_bytes[b] / 16; v += 32) r[v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Exact three-term bf16 split of an fp32 value (Henry, Tang and Heinecke 2019):
// v = hi + mid + lo with hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid).
__device__ __forceinline__ void split3(float v, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

__global__ void __launch_bounds__(256) k_split_grad(const float* __restrict__ dl, const float* __restrict__ dn,
                                                    int T, int E, int E8, int nblk, __nv_bfloat16* __restrict__ out)
{
    griddep_launch_dependents();
    griddep_wait();
    const int W = nblk * E8;
    const long long total = (long long)T * W;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / W), c = (int)(i - (long long)t * W);
        const int blk = c / E8, e = c - blk * E8;
        const float* src = blk < 4 ? dl : dn;
        const float v = e < E ? src[(size_t)t * E + e] : 0.0f;
        __nv_bfloat16 hi, mid, lo;
        split3(v, hi, mid, lo);
        const int term = blk & 3;  // hi, mid, lo, hi
        out[i] = term == 1 ? mid : (term == 2 ? lo : hi);
    }
}

__global__ void __launch_bounds__(256) k_split_wcat(const float* __restrict__ Wg, const float* __restrict__ Wn,
                                                    int E, int E8, int d, int nblk, __nv_bfloat16* __restrict__ out)
{
    griddep_launch_dependents();
    griddep_wait();
    const long long total = (long long)nblk * E8 * d;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(i / d), col = (int)(i - (long long)r * d);
        const int blk = r / E8, e = r - blk * E8;
        const float* src = blk < 4 ? Wg : Wn;
        const float v = e < E ? src[(size_t)e * d + col] : 0.0f;
        __nv_bfloat16 hi, mid, lo;
        split3(v, hi, mid, lo);
        out[i] = (blk & 3) == 3 ? mid : hi;  // hi, hi, hi, mid
    }
}

__global__ void __launch_bounds__(256) k_sum3(const float* __restrict__ P, int splits, int E, int E8, int d,
                                              float* __restrict__ out)
{
    griddep_launch_dependents();
    griddep_wait();
    const long long total = (long long)E * d;
    const long long blk = (long long)E8 * d;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (int sp = 0; sp < splits; ++sp) {
            const float* p = P + (long long)sp * 3 * blk;
            acc += (p[2 * blk + i] + p[blk + i]) + p[i];  // smallest terms first
        }
        out[i] = acc;
    }
}

int elem_grid(long long n, int sms)
{
    long long g = (n + 255) / 256;
    if (g > (long long)sms * 16) g = (long long)sms * 16;
    return (int)(g < 1 ? 1 : g);
}

int warp_grid(int T, int sms)
{
    const int g = ceil_div(T, 8);
    return g < sms * 16 ? g : sms * 16;
}

}  // namespace

cudaError_t launch_bwd_combine(const BwdCombineArgs& a, bool bf16, int sms, cudaStream_t st, bool pdl)
{
    const dim3 grid(warp_grid(a.T, sms)), block(256);
    if (bf16) return launch_kernel(k_bwd_combine<__nv_bfloat16>, grid, block, 0, st, pdl, a);
    return launch_kernel(k_bwd_combine<float>, grid, block, 0, st, pdl, a);
}

cudaError_t launch_router_bwd(const RouterBwdArgs& a, int sms, cudaStream_t st, bool pdl)
{
    const dim3 grid(warp_grid(a.T, sms)), block(256);
    if (a.E <= 32) return launch_kernel(k_router_bwd<1>, grid, block, 0, st, pdl, a);
    if (a.E <= 64) return launch_kernel(k_router_bwd<2>, grid, block, 0, st, pdl, a);
    if (a.E <= 128) return launch_kernel(k_router_bwd<4>, grid, block, 0, st, pdl, a);
    if (a.E <= 256) return launch_kernel(k_router_bwd<8>, grid, block, 0, st, pdl, a);
    return launch_kernel(k_router_bwd<16>, grid, block, 0, st, pdl, a);
}

cudaError_t launch_colsum(const ColsumArgs& a, int types, int sms, cudaStream_t st, bool pdl)
{
    long long grid = (long long)a.G * ceil_div(a.N, 32);
    if (grid > (long long)sms * 8) grid = (long long)sms * 8;
    if (grid < 1) grid = 1;
    const dim3 g((int)grid), b(256);
    switch (types) {
    case kBwdTypesBf16: return launch_kernel(k_colsum<__nv_bfloat16, __nv_bfloat16>, g, b, 0, st, pdl, a);
    default: return launch_kernel(k_colsum<float, float>, g, b, 0, st, pdl, a);
    }
}

cudaError_t launch_split_grad(const float* dl, const float* dn, int T, int E, int E8, int nblk, void* out,
                              int sms, cudaStream_t st, bool pdl)
{
    return launch_kernel(k_split_grad, dim3(elem_grid((long long)T * nblk * E8, sms)), dim3(256), 0, st, pdl, dl, dn,
                         T, E, E8, nblk, static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_split_wcat(const float* Wg, const float* Wn, int E, int E8, int d, int nblk, void* out,
                              int sms, cudaStream_t st, bool pdl)
{
    return launch_kernel(k_split_wcat, dim3(elem_grid((long long)nblk * E8 * d, sms)), dim3(256), 0, st, pdl, Wg,
                         Wn, E, E8, d, nblk, static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_sum3(const float* P, int splits, int E, int E8, int d, float* out, int sms, cudaStream_t st,
                        bool pdl)
{
    return launch_kernel(k_sum3, dim3(elem_grid((long long)E * d, sms)), dim3(256), 0, st, pdl, P, splits, E, E8, d,
                         out);
}

int router_dw_splits(int T, int E8, int d)
{
    const int tiles = ceil_div(3 * E8, 128) * ceil_div(d, 256);
    int s = 1;
    while (s < 16 && tiles * s * 2 <= 148 && ceil_div(T, s * 2) >= 256) s *= 2;
    return s;
}

cudaError_t launch_zero_pad_rows(const ZeroPadArgs& a, int sms, cudaStream_t st, bool pdl)
{
    const dim3 grid(warp_grid(a.G * 64, sms)), block(256);
    return launch_kernel(k_zero_pad_rows, grid, block, 0, st, pdl, a);
}

cudaError_t launch_bwd_unpermute(const BwdUnpermuteArgs& a, bool bf16, int sms, cudaStream_t st, bool pdl)
{
    const dim3 grid(warp_grid(a.T, sms)), block(256);
    if (bf16) return launch_kernel(k_bwd_unpermute<__nv_bfloat16>, grid, block, 0, st, pdl, a);
    return launch_kernel(k_bwd_unpermute<float>, grid, block, 0, st, pdl, a);
}

}  // namespace moe
