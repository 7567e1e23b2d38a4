// combine.cu -- stage 4 of the layer: gate-weighted un-permute and accumulate.
//
// y[t] = sum over the kept slots j of token t (slot order) of g[t,j] * Yp[row(t,j)]
//      + Ys[t]                (shared experts, gate 1; "MoE 混合专家模型串讲" §"共享专家隔离")
//      + x[t] if pass(t)      (dropped token: 0 + x = x; "MoE 混合专家模型串讲" §"专家容量")
// accumulated in fp32 and rounded once ("混合专家模型MoE入门实战" §3.4 output[mask]
// += weight * expert_output; "混合专家 MOE 是什么" y = sum_i g_i e_i(x)).
// pass(t) is 1 for every token when residual_mode == 1; with residual_mode 0 it
// is 1 only when all k routed slots of t were dropped.
//
// One warp per (token, row segment); each lane handles 16-byte vectors of the
// row; no atomics, so the result is deterministic.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <typename T, bool SEG>
__global__ void __launch_bounds__(256) k_combine(CombineArgs a)
{
    constexpr int V = Vec<T>::N;
    __shared__ int s_row[8][kMaxTopK];
    __shared__ float s_gate[8][kMaxTopK];
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = a.d / V;
    const int seg = SEG ? a.seg_vec : nvec;  // 16-byte vectors per work item
    const int nseg = SEG ? ceil_div(nvec, seg) : 1;
    const int items = a.T * nseg;  // < 2^31: nseg > 1 only for T < 8192
    const size_t row_bytes = (size_t)a.d * sizeof(T);
    const unsigned all_k = (a.k >= 32) ? 0xffffffffu : ((1u << a.k) - 1u);

    // work item = (token, segment of the row): whole rows for large batches, several
    // independent warps per token when the batch is small
    for (int item = blockIdx.x * 8 + warp; item < items; item += gridDim.x * 8) {
        const int t = item / nseg;
        const int v0 = (item - t * nseg) * seg;
        const int v1 = min(nvec, v0 + seg);
        int r = -1;
        float g = 0.0f;
        if (lane < a.k) {
            r = a.slot_row[(size_t)t * a.k + lane];
            g = a.gates[(size_t)t * a.k + lane];
            s_row[warp][lane] = r;
            s_gate[warp][lane] = g;
        }
        const unsigned dropped = __ballot_sync(0xffffffffu, lane < a.k && r < 0);
        const bool pass = a.residual_mode == 1 || dropped == all_k;
        __syncwarp();
        const char* xrow = static_cast<const char*>(a.x) + (size_t)t * row_bytes;
        const char* ysrow = a.ys ? static_cast<const char*>(a.ys) + (size_t)t * row_bytes : nullptr;
        char* yrow = static_cast<char*>(a.y) + (size_t)t * row_bytes;
        for (int v = v0 + lane; v < v1; v += 32) {
            float acc[V];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = 0.0f;
            for (int j = 0; j < a.k; ++j) {
                const int rj = s_row[warp][j];
                if (rj < 0) continue;
                const float gj = s_gate[warp][j];
                float u[V];
                Vec<T>::load(static_cast<const char*>(a.yp) + (size_t)rj * row_bytes + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = fmaf(gj, u[i], acc[i]);
            }
            if (ysrow) {
                float u[V];
                Vec<T>::load(ysrow + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += u[i];
            }
            if (pass) {
                float u[V];
                Vec<T>::load(xrow + v * 16, u);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += u[i];
            }
            Vec<T>::store(yrow + v * 16, acc);
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool bf16, int num_sms, cudaStream_t st, bool pdl)
{
    // one warp per token keeps the GPU full from about 8192 tokens on; smaller batches
    // split each row into segments (multiples of 32 vectors) to raise the warp count
    const int nvec = a.d / (bf16 ? 8 : 4);
    int nseg = a.T >= 8192 ? 1 : ceil_div(16384, a.T);
    const int max_seg = ceil_div(nvec, 32);
    if (nseg > max_seg) nseg = max_seg;
    CombineArgs b = a;
    b.seg_vec = ceil_div(ceil_div(nvec, nseg), 32) * 32;
    const long long items = (long long)a.T * ceil_div(nvec, b.seg_vec);
    long long grid = (items + 7) / 8;
    if (grid > (long long)num_sms * 32) grid = (long long)num_sms * 32;
    const dim3 g((int)grid), blk(256);
    if (ceil_div(nvec, b.seg_vec) > 1) {
        if (bf16) return launch_kernel(k_combine<__nv_bfloat16, true>, g, blk, 0, st, pdl, b);
        return launch_kernel(k_combine<float, true>, g, blk, 0, st, pdl, b);
    }
    if (bf16) return launch_kernel(k_combine<__nv_bfloat16, false>, g, blk, 0, st, pdl, b);
    return launch_kernel(k_combine<float, false>, g, blk, 0, st, pdl, b);
}

}  // namespace moe
