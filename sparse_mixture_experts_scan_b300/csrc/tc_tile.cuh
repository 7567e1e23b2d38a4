// tc_tile.cuh -- pieces shared by the tcgen05 GEMM kernels: the grouped tile
// map, the accumulator epilogue (TMEM -> registers -> activation -> bf16 -> global)
// and the short drain wait.
#pragma once

#include "common.cuh"

namespace moe {

// Tiles of a grouped GEMM: group g owns M-tiles mt[g] .. mt[g+1]-1; each M-tile has
// n_tiles N-tiles; inside a group the tile index runs M fastest, so consecutive tiles
// share the B (weight) tile.
struct TileMap {
    int g = 0;
    // Advance to the group holding `tile` (tiles are visited in increasing order).
    __device__ __forceinline__ void locate(int tile, const int* mt, int n_tiles, int& m, int& n)
    {
        while (tile >= mt[g + 1] * n_tiles) ++g;
        const int local = tile - mt[g] * n_tiles;
        const int mtg = mt[g + 1] - mt[g];
        n = local / mtg;
        m = local - n * mtg;
    }
};

// Round 32 consecutive outputs of one row to bf16 and store the 16-byte groups
// that lie inside the N valid columns (N is a multiple of 8).
__device__ __forceinline__ void store_row32(__nv_bfloat16* orow, int col0, int N, const float (&o)[32])
{
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int col = col0 + v * 8;
        if (col + 8 <= N) {
            uint4 u;
            u.x = pack_bf16x2(o[v * 8 + 0], o[v * 8 + 1]);
            u.y = pack_bf16x2(o[v * 8 + 2], o[v * 8 + 3]);
            u.z = pack_bf16x2(o[v * 8 + 4], o[v * 8 + 5]);
            u.w = pack_bf16x2(o[v * 8 + 6], o[v * 8 + 7]);
            *reinterpret_cast<uint4*>(orow + col) = u;
        }
    }
}

// One thread = one accumulator row (its TMEM lane).  Reads the accumulator columns,
// applies bias and activation (or pairs the W1 half [0, BN/2) with the W3 half
// [BN/2, BN) for SwiGLU) and stores bf16 outputs n0 .. n0 + OUT_COLS - 1 of the row.
// The bias of column c is sum over K-segments sg of bias[bias_base + sg * seg_stride + c].
// Every thread of the warp must call it (tcgen05.ld is warp-collective).
// SAVE: also store the pre-activations (training): z1 = the W1 half (+ bias), z3 =
// the W3 half, rows laid out like orow.
template <int BN, int ACT, bool SAVE = false>
__device__ __forceinline__ void epilogue_tile(uint32_t t_lane, __nv_bfloat16* orow, bool row_ok, int n0, int N,
                                              const __nv_bfloat16* bias, size_t bias_base, int k_segments,
                                              int seg_stride, __nv_bfloat16* z1row = nullptr,
                                              __nv_bfloat16* z3row = nullptr)
{
    constexpr bool GATED = (ACT == kActSwiglu);
    constexpr int OUT_COLS = GATED ? BN / 2 : BN;
    if constexpr (GATED) {
#pragma unroll 1
        for (int c = 0; c < OUT_COLS / 32; ++c) {
            uint32_t va[32], vb[32];
            tmem_ld_32cols(t_lane + c * 32, va);
            tmem_ld_32cols(t_lane + BN / 2 + c * 32, vb);
            tmem_ld_wait();
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                o[i] = activate_bf16out<kActSwiglu>(__uint_as_float(va[i])) * __uint_as_float(vb[i]);
            if (row_ok) store_row32(orow, n0 + c * 32, N, o);
            if constexpr (SAVE) {
                if (row_ok) {
                    store_row32(z1row, n0 + c * 32, N, reinterpret_cast<const float(&)[32]>(va));
                    store_row32(z3row, n0 + c * 32, N, reinterpret_cast<const float(&)[32]>(vb));
                }
            }
        }
    } else if (bias == nullptr) {
#pragma unroll 1
        for (int c = 0; c < OUT_COLS / 32; ++c) {
            uint32_t va[32];
            tmem_ld_32cols(t_lane + c * 32, va);
            tmem_ld_wait();
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = activate_bf16out<ACT>(__uint_as_float(va[i]));
            if (row_ok) store_row32(orow, n0 + c * 32, N, o);
            if constexpr (SAVE) {
                if (row_ok) store_row32(z1row, n0 + c * 32, N, reinterpret_cast<const float(&)[32]>(va));
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < OUT_COLS / 32; ++c) {
            uint32_t va[32];
            tmem_ld_32cols(t_lane + c * 32, va);
            tmem_ld_wait();
            float bsum[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) bsum[i] = 0.0f;
            const int col0 = n0 + c * 32;
            for (int sg = 0; sg < k_segments; ++sg) {
                const __nv_bfloat16* bp = bias + bias_base + (size_t)sg * seg_stride;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (col0 + i < N) bsum[i] += __bfloat162float(bp[col0 + i]);
            }
            float o[32], z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                z[i] = __uint_as_float(va[i]) + bsum[i];
                o[i] = activate_bf16out<ACT>(z[i]);
            }
            if (row_ok) store_row32(orow, col0, N, o);
            if constexpr (SAVE) {
                if (row_ok) store_row32(z1row, col0, N, z);
            }
        }
    }
}

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ bool mbar_wait_short(uint64_t* bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 100000000ull) return false;  // 100 ms
    return true;
}

}  // namespace moe
