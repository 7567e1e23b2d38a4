// gemm_bwd_ffma.cu -- the grouped GEMMs of the backward pass on the CUDA cores.
//
// One strided kernel covers every product of the backward (BwdGemmArgs):
//   dgrad  (rows of expert segment g):  dH = dYp W2_e,  dXp = dZ1 W1_e (+ dZ3 W3_e)
//   wgrad  (reduction over segment g):  dW2_e = dYp_e^T H_e,  dW1_e = dZ1_e^T Xp_e, ...
//   fixed  (one group):                 router and shared-expert products
// with the activation backward fused into the dgrad of the second layer.  It is
// the fp32 path and, for bf16 layers, the cross-check of the tensor-core path.
//
// Tile: 128 rows x 64 columns, K-steps of 16 through shared memory; 256 threads,
// each owns 8 rows x 4 columns; persistent over the tile list.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTM = 128, kTN = 64, kTK = 16;

template <typename T>
__device__ __forceinline__ void store_out(T* p, float v)
{
    if constexpr (sizeof(T) == 2) *p = __float2bfloat16_rn(v);
    else *p = v;
}

template <typename TA, typename TB, typename TC, int EPI>
__global__ void __launch_bounds__(256) k_gemm_bwd_ffma(BwdGemmArgs a)
{
    __shared__ float As[kTK][kTM + 4];
    __shared__ float Bs[kTK][kTN + 4];
    __shared__ int s_mt[kMaxExperts + 1];

    griddep_launch_dependents();
    griddep_wait();
    const int G = a.mode == kBwdFixed ? 1 : a.G;
    const int n_tiles = ceil_div(a.N, kTN);
    // M-tiles per group: from the device prefix for row-grouped products, else fixed
    for (int i = threadIdx.x; i <= G; i += 256)
        s_mt[i] = a.mode == kBwdRows ? a.mtile_off[i] : i * ceil_div(a.M, kTM);
    __syncthreads();

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int total = s_mt[G] * n_tiles;
    const TA* A = static_cast<const TA*>(a.A);
    const TB* B = static_cast<const TB*>(a.B);
    const TA* A2 = static_cast<const TA*>(a.A2);
    const TB* B2 = static_cast<const TB*>(a.B2);
    TC* C = static_cast<TC*>(a.C);

    int g = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        while (tile >= s_mt[g + 1] * n_tiles) ++g;
        const int local = tile - s_mt[g] * n_tiles;
        const int mtg = s_mt[g + 1] - s_mt[g];
        const int n = local / mtg, m = local - n * mtg;
        // extents and operand bases of group g
        long long a_base = 0, b_base = (long long)(a.b_g0 + g) * a.b_gs, c_base = 0;
        int Mg = a.M, Kg = a.K;
        if (a.mode == kBwdRows) {
            a_base = (long long)a.row_off[g] * a.a_sm;
            c_base = (long long)a.row_off[g] * a.c_sm;
            Mg = a.rows[g];
        } else if (a.mode == kBwdReduce) {
            a_base = (long long)a.row_off[g] * a.a_sk;
            b_base = (long long)a.row_off[g] * a.b_sk;
            c_base = (long long)(a.c_g0 + g) * a.c_gs;
            Kg = a.rows[g];
        }
        const int m0 = m * kTM, n0 = n * kTN;

        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

        for (int seg = 0; seg < (A2 != nullptr ? 2 : 1); ++seg) {
            const TA* Ap = seg == 0 ? A : A2;
            const TB* Bp = seg == 0 ? B : B2;
            for (int k0 = 0; k0 < Kg; k0 += kTK) {
                // A tile 128 x 16: element (m, k) at a_base + m*a_sm + k*a_sk
                for (int v = tid; v < kTM * kTK; v += 256) {
                    int r, c;
                    if (a.a_sk == 1) {  // k contiguous: consecutive threads walk k
                        r = v / kTK;
                        c = v % kTK;
                    } else {            // m contiguous
                        c = v / kTM;
                        r = v % kTM;
                    }
                    const int gm = m0 + r, gk = k0 + c;
                    As[c][r] = (gm < Mg && gk < Kg)
                                   ? to_f32(Ap[a_base + (long long)gm * a.a_sm + (long long)gk * a.a_sk])
                                   : 0.0f;
                }
                // B tile 16 x 64: element (k, n) at b_base + k*b_sk + n*b_sn
                for (int v = tid; v < kTK * kTN; v += 256) {
                    int r, c;
                    if (a.b_sn == 1) {
                        r = v / kTN;
                        c = v % kTN;
                    } else {
                        c = v / kTK;
                        r = v % kTK;
                    }
                    const int gk = k0 + r, gn = n0 + c;
                    Bs[r][c] = (gk < Kg && gn < a.N)
                                   ? to_f32(Bp[b_base + (long long)gk * a.b_sk + (long long)gn * a.b_sn])
                                   : 0.0f;
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < kTK; ++kk) {
                    float av[8], bv[4];
#pragma unroll
                    for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
                }
                __syncthreads();
            }
        }

#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int gm = m0 + ty * 8 + i;
            if (gm >= Mg) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gn = n0 + tx * 4 + j;
                if (gn >= a.N) continue;
                const long long o = c_base + (long long)gm * a.c_sm + gn;
                const float v = acc[i][j];
                if constexpr (EPI == kEpiStore) {
                    const float b = a.bias != nullptr
                                        ? to_f32(static_cast<const TC*>(a.bias)[(long long)(a.b_g0 + g) * a.N + gn])
                                        : 0.0f;
                    store_out(C + o, v + b);
                } else if constexpr (EPI == kEpiReluBwd) {
                    // relu'(z) from the saved output h = relu(z): 1 where h > 0
                    store_out(C + o, to_f32(static_cast<const TC*>(a.e1)[o]) > 0.0f ? v : 0.0f);
                } else if constexpr (EPI == kEpiSwigluBwd) {
                    const float z1 = to_f32(static_cast<const TC*>(a.e1)[o]);
                    const float z3 = to_f32(static_cast<const TC*>(a.e2)[o]);
                    store_out(C + o, v * z3 * silu_grad_f32(z1));
                    store_out(static_cast<TC*>(a.C2) + o, v * silu_f32(z1));
                } else {
                    const float z = to_f32(static_cast<const TC*>(a.e1)[o]);
                    store_out(C + o, v * act_grad_f32<EPI == kEpiGeluTanhBwd ? kActGeluTanh : kActGeluErf>(z));
                }
            }
        }
    }
}

template <typename TA, typename TB, typename TC>
cudaError_t launch_t(const BwdGemmArgs& a, int grid, cudaStream_t st, bool pdl)
{
    switch (a.epi) {
    case kEpiStore: return launch_kernel(k_gemm_bwd_ffma<TA, TB, TC, kEpiStore>, dim3(grid), dim3(256), 0, st, pdl, a);
    case kEpiReluBwd:
        return launch_kernel(k_gemm_bwd_ffma<TA, TB, TC, kEpiReluBwd>, dim3(grid), dim3(256), 0, st, pdl, a);
    case kEpiGeluTanhBwd:
        return launch_kernel(k_gemm_bwd_ffma<TA, TB, TC, kEpiGeluTanhBwd>, dim3(grid), dim3(256), 0, st, pdl, a);
    case kEpiGeluErfBwd:
        return launch_kernel(k_gemm_bwd_ffma<TA, TB, TC, kEpiGeluErfBwd>, dim3(grid), dim3(256), 0, st, pdl, a);
    default: return launch_kernel(k_gemm_bwd_ffma<TA, TB, TC, kEpiSwigluBwd>, dim3(grid), dim3(256), 0, st, pdl, a);
    }
}

}  // namespace

cudaError_t launch_gemm_bwd_ffma(const BwdGemmArgs& a, int types, int grid, cudaStream_t st, bool pdl)
{
    switch (types) {
    case kBwdTypesBf16: return launch_t<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(a, grid, st, pdl);
    case kBwdTypesF32: return launch_t<float, float, float>(a, grid, st, pdl);
    default:  // kBwdTypesF32xBf16: router products with fp32 gradients and bf16 x (plain stores)
        return launch_kernel(k_gemm_bwd_ffma<float, __nv_bfloat16, float, kEpiStore>, dim3(grid), dim3(256), 0, st,
                             pdl, a);
    }
}

}  // namespace moe
