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

// One warp per token.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_combine(BwdCombineArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* dy = static_cast<const T*>(a.dy);
    const T* yp = static_cast<const T*>(a.yp);
    T* dyp = static_cast<T*>(a.dyp);
    for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
        const T* dyr = dy + (size_t)t * a.d;
        for (int j = 0; j < a.k; ++j) {
            const size_t s = (size_t)t * a.k + j;
            const int r = a.slot_row[s];
            float dot = 0.0f;
            if (r >= 0) {
                const float g = a.gates[s];
                const T* yr = yp + (size_t)r * a.d;
                T* dr = dyp + (size_t)r * a.d;
                for (int i = lane; i < a.d; i += 32) {
                    const float v = ld_f32(dyr, i);
                    dot = fmaf(v, ld_f32(yr, i), dot);
                    st_round(dr, i, g * v);
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

// out[g][n] = sum over the rows of segment g of A[row][n]; one thread per (g, n).
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) k_colsum(ColsumArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const TI* A = static_cast<const TI*>(a.A);
    TO* out = static_cast<TO*>(a.out);
    const long long total = (long long)a.G * a.N;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int g = (int)(i / a.N), n = (int)(i - (long long)g * a.N);
        const long long r0 = a.row_off != nullptr ? a.row_off[g] : 0;
        const int rows = a.rows != nullptr ? a.rows[g] : a.fixed_rows;
        float s = 0.0f;
        for (int r = 0; r < rows; ++r) s += to_f32(A[(r0 + r) * a.lda + n]);
        st_round(out, (size_t)(a.out_g0 + g) * a.N + n, s);
    }
}

// One warp per token, d elements per row, fp32 accumulation in a fixed order.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_unpermute(BwdUnpermuteArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* dy = static_cast<const T*>(a.dy);
    const T* dxp = static_cast<const T*>(a.dxp);
    const T* dxs = static_cast<const T*>(a.dxs);
    T* dx = static_cast<T*>(a.dx);
    for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
        int n_drop = 0;
        for (int j = 0; j < a.k; ++j) n_drop += a.slot_row[(size_t)t * a.k + j] < 0 ? 1 : 0;
        const bool pass = a.residual_mode == 1 || n_drop == a.k;
        for (int i = lane; i < a.d; i += 32) {
            float v = pass ? ld_f32(dy, (size_t)t * a.d + i) : 0.0f;
            for (int j = 0; j < a.k; ++j) {
                const int r = a.slot_row[(size_t)t * a.k + j];
                if (r >= 0) v += ld_f32(dxp, (size_t)r * a.d + i);
            }
            if (dxs != nullptr) v += ld_f32(dxs, (size_t)t * a.d + i);
            v += a.dxr[(size_t)t * a.d + i];
            st_round(dx, (size_t)t * a.d + i, v);
        }
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
    const long long total = (long long)a.G * a.N;
    long long grid = (total + 255) / 256;
    if (grid > (long long)sms * 8) grid = (long long)sms * 8;
    if (grid < 1) grid = 1;
    const dim3 g((int)grid), b(256);
    switch (types) {
    case kBwdTypesBf16: return launch_kernel(k_colsum<__nv_bfloat16, __nv_bfloat16>, g, b, 0, st, pdl, a);
    default: return launch_kernel(k_colsum<float, float>, g, b, 0, st, pdl, a);
    }
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
