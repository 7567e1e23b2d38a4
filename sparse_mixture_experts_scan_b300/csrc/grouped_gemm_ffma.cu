// grouped_gemm_ffma.cu -- stage 3 of the layer on the CUDA cores (FFMA).
//
// Same grouped problem as grouped_gemm_tc.cu (see GroupedGemmArgs): per expert
// segment, out = act(A B^T (+ bias)), or the SwiGLU pairing silu(A W1^T) *
// (A W3^T).  Used for fp32 layers (fp32 accuracy; tensor-core TF32 would not
// meet an fp32 tolerance) and, for bf16 layers, as a cross-check kernel.
//
// Tile: 128 rows x 64 output columns, K-steps of 16 staged in shared memory;
// 256 threads, each owns 8 rows x 4 columns; persistent over the tile list.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTM = 128, kTN = kFfmaTileN, kTK = 16;

template <typename T, int ACT>
__global__ void __launch_bounds__(256) k_grouped_gemm_ffma(const T* __restrict__ A, int lda,
                                                           const T* __restrict__ B,
                                                           const T* __restrict__ B3, int ldb,
                                                           GroupedGemmArgs args)
{
    constexpr bool GATED = (ACT == kActSwiglu);
    __shared__ float As[kTK][kTM + 4];
    __shared__ float Bs[kTK][kTN + 4];
    __shared__ float B3s[GATED ? kTK : 1][kTN + 4];
    __shared__ int s_mt[kMaxExperts + 1];

    griddep_launch_dependents();
    griddep_wait();
    const bool fixed = args.mtile_off == nullptr;
    const int G = fixed ? 1 : args.G;
    for (int i = threadIdx.x; i <= G; i += 256)
        s_mt[i] = fixed ? (i == 0 ? 0 : ceil_div(args.fixed_rows, kTM)) : args.mtile_off[i];
    __syncthreads();

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;  // rows ty*8.., cols tx*4..
    const int n_tiles = args.n_tiles;
    const int total = s_mt[G] * n_tiles;
    T* out = static_cast<T*>(args.out);
    const T* bias = static_cast<const T*>(args.bias);

    int g = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        while (tile >= s_mt[g + 1] * n_tiles) ++g;
        const int local = tile - s_mt[g] * n_tiles;
        const int mtg = s_mt[g + 1] - s_mt[g];
        const int n = local / mtg, m = local - n * mtg;
        const int row0 = (fixed ? 0 : args.row_off[g]) + m * kTM;  // row in A / out
        const int rows_g = fixed ? args.fixed_rows : args.rows[g];
        const int n0 = n * kTN;

        float acc[8][4], acc3[GATED ? 8 : 1][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = 0.0f;
                if (GATED) acc3[GATED ? i : 0][j] = 0.0f;
            }

        for (int sg = 0; sg < args.k_segments; ++sg) {
            const size_t b_base = (size_t)(args.b_group0 + g + sg) * args.b_rows_per_group;
            for (int k0 = 0; k0 < args.K; k0 += kTK) {
                // A: 128 x 16 -> As[k][row]; thread loads 8 consecutive k of one row
                {
                    const int r = tid / 2, c0 = (tid % 2) * 8;
                    const int grow = row0 + r;
                    for (int c = 0; c < 8; ++c) {
                        const int kk = k0 + c0 + c;
                        float v = 0.0f;
                        if (grow < args.a_rows_alloc && kk < args.K)
                            v = to_f32(A[(size_t)grow * lda + (size_t)sg * args.K + kk]);
                        As[c0 + c][r] = v;
                    }
                }
                // B (and W3): 64 x 16 -> Bs[k][col]; thread loads 4 consecutive k of one row
                {
                    const int r = tid / 4, c0 = (tid % 4) * 4;
                    const int ncol = n0 + r;
                    for (int c = 0; c < 4; ++c) {
                        const int kk = k0 + c0 + c;
                        const bool ok = ncol < args.N && kk < args.K;
                        const size_t off = (b_base + ncol) * ldb + kk;
                        Bs[c0 + c][r] = ok ? to_f32(B[off]) : 0.0f;
                        if (GATED) B3s[GATED ? c0 + c : 0][r] = ok ? to_f32(B3[off]) : 0.0f;
                    }
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < kTK; ++kk) {
                    float av[8], bv[4], b3v[4];
#pragma unroll
                    for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        bv[j] = Bs[kk][tx * 4 + j];
                        if (GATED) b3v[j] = B3s[GATED ? kk : 0][tx * 4 + j];
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
                            if (GATED) acc3[GATED ? i : 0][j] = fmaf(av[i], b3v[j], acc3[GATED ? i : 0][j]);
                        }
                }
                __syncthreads();
            }
        }

#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = m * kTM + ty * 8 + i;  // row inside the group
            if (r >= rows_g) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = n0 + tx * 4 + j;
                if (col >= args.N) continue;
                float z = acc[i][j];
                float o;
                if constexpr (GATED) {
                    o = activate<kActSwiglu>(z) * acc3[i][j];
                } else {
                    if (bias != nullptr)
                        for (int sg = 0; sg < args.k_segments; ++sg)
                            z += to_f32(bias[(size_t)(args.b_group0 + g + sg) * args.b_rows_per_group + col]);
                    o = activate<ACT>(z);
                }
                if constexpr (sizeof(T) == 2) out[(size_t)(row0 + ty * 8 + i) * args.ldo + col] = __float2bfloat16_rn(o);
                else out[(size_t)(row0 + ty * 8 + i) * args.ldo + col] = o;
            }
        }
    }
}

template <typename T>
cudaError_t launch_ffma_t(const void* A, int lda, const void* B, const void* B3, int ldb,
                          const GroupedGemmArgs& args, int act, int grid, cudaStream_t st, bool pdl)
{
    const T* a = static_cast<const T*>(A);
    const T* b = static_cast<const T*>(B);
    const T* b3 = static_cast<const T*>(B3);
    switch (act) {
    case kActNone: return launch_kernel(k_grouped_gemm_ffma<T, kActNone>, dim3(grid), dim3(256), 0, st, pdl, a, lda, b, b3, ldb, args);
    case kActRelu: return launch_kernel(k_grouped_gemm_ffma<T, kActRelu>, dim3(grid), dim3(256), 0, st, pdl, a, lda, b, b3, ldb, args);
    case kActGeluTanh: return launch_kernel(k_grouped_gemm_ffma<T, kActGeluTanh>, dim3(grid), dim3(256), 0, st, pdl, a, lda, b, b3, ldb, args);
    case kActGeluErf: return launch_kernel(k_grouped_gemm_ffma<T, kActGeluErf>, dim3(grid), dim3(256), 0, st, pdl, a, lda, b, b3, ldb, args);
    default: return launch_kernel(k_grouped_gemm_ffma<T, kActSwiglu>, dim3(grid), dim3(256), 0, st, pdl, a, lda, b, b3, ldb, args);
    }
}

}  // namespace

cudaError_t launch_gemm_ffma(const void* A, int lda, const void* B, const void* B3, int ldb,
                             const GroupedGemmArgs& args, int act, bool bf16, int grid, cudaStream_t st, bool pdl)
{
    if (bf16) return launch_ffma_t<__nv_bfloat16>(A, lda, B, B3, ldb, args, act, grid, st, pdl);
    return launch_ffma_t<float>(A, lda, B, B3, ldb, args, act, grid, st, pdl);
}

}  // namespace moe
