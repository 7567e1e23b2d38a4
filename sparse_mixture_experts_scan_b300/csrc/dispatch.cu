// dispatch.cu -- stage 2 of the layer: token-order capacity and the row permute.
//
// "混合专家模型MoE入门实战" §2.4: tokens that chose the same expert are gathered
// together, run as one batch, and scattered back.  Here the gather is a
// histogram + device-wide scan, and a permute of token rows into one buffer
// where every expert owns a contiguous segment padded to kSegRows rows.
//
// Capacity ("MoE架构解析" §3.1 expert_capacity = int(T * cf / E); "MoE 混合专家
// 模型串讲" §"专家容量"): the slots of each expert are ranked in token order;
// rank >= C is dropped (the token skips that expert, f(x) = 0).
//
// k_dispatch_scan: one block per chunk of 1024 slots (slot s = t*k + j, so
// slot order is token order and a token never picks one expert twice).
//   - warp rank of each slot among equal experts: __match_any_sync;
//   - per-warp histogram in shared memory, scanned over the 32 warps in order:
//     the slot's rank inside its chunk;
//   - the last block to arrive scans the chunk histograms per expert (counts,
//     chunk bases), the per-expert kept counts over experts (segment offsets,
//     M-tile offsets for the grouped GEMM).
// The balance statistic is reduced in two levels: every scan block sums a slice
// of the router's per-block probability sums, the last block adds those partials.
// k_permute: one warp per slot; position = chunk base + rank; kept rows are
// copied with 16-byte vector loads/stores.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Exclusive scan of three ints over the 1024 threads of a block, in thread order.
__device__ void block_exclusive_scan3(const int (&v)[3], int (&out)[3], int (&total)[3],
                                      int (*wsum)[3])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int u = __shfl_up_sync(0xffffffffu, inc[q], o);
            if (lane >= o) inc[q] += u;
        }
    }
    if (lane == 31)
#pragma unroll
        for (int q = 0; q < 3; ++q) wsum[warp][q] = inc[q];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            int w = wsum[lane][q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += u;
            }
            wsum[lane][q] = w;
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        out[q] = (warp > 0 ? wsum[warp - 1][q] : 0) + inc[q] - v[q];
        total[q] = wsum[31][q];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(1024) k_dispatch_scan(DispatchArgs a)
{
    extern __shared__ int32_t sm[];  // [32][E] warp histograms, reused by the last block
    __shared__ int wsum[32][3];
    __shared__ double dsum[32];
    __shared__ int s_last;

    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E;
    const long long n_slots = (long long)a.T * a.k;
    const long long s = (long long)blockIdx.x * kScanChunk + tid;
    // an index outside [0, E) (never produced by the router; possible in caller-provided
    // indices) is not counted and its slot ends up dropped
    int e = s < n_slots ? a.idx[s] : -1;
    if (e < 0 || e >= E) e = -1;
    const bool valid = e >= 0;

    for (int i = tid; i < 32 * E; i += 1024) sm[i] = 0;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int wrank = __popc(peers & ((1u << lane) - 1u));
    if (valid && wrank == 0) sm[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += 1024) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int v = sm[w * E + ee];
            sm[w * E + ee] = run;
            run += v;
        }
        a.chunk_hist[(size_t)blockIdx.x * E + ee] = run;
    }
    __syncthreads();
    if (valid) a.local_rank[s] = sm[warp * E + e] + wrank;

    // balance statistic, first level: this block sums a contiguous slice of the
    // router's per-block column sums (fixed order: partition p takes rows r0+p,
    // r0+p+P, ...; partitions added in order)
    const int P = 1024 / E;
    if (a.n_router_blocks > 0) {
        __syncthreads();  // sm is reused below
        float* s_part = reinterpret_cast<float*>(sm);
        const int R = a.n_router_blocks, nb = gridDim.x;
        const int r0 = (int)((long long)blockIdx.x * R / nb);
        const int r1 = (int)((long long)(blockIdx.x + 1) * R / nb);
        if (tid < P * E) {
            const int ee = tid % E, p = tid / E;
            float acc = 0.0f;
            int r = r0 + p;
            // up to 16 loads in flight per thread (one or two memory round trips for the
            // few hundred rows a block sums), added in order
            for (; r + 15 * P < r1; r += 16 * P) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = __ldcg(&a.psum_part[(size_t)(r + u * P) * E + ee]);
#pragma unroll
                for (int u = 0; u < 16; ++u) acc += v[u];
            }
            for (; r + 3 * P < r1; r += 4 * P) {
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = __ldcg(&a.psum_part[(size_t)(r + u * P) * E + ee]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc += v[u];
            }
            for (; r < r1; r += P) acc += __ldcg(&a.psum_part[(size_t)r * E + ee]);
            s_part[p * E + ee] = acc;
        }
        __syncthreads();
        if (tid < E) {
            float acc = 0.0f;
            for (int p = 0; p < P; ++p) acc += s_part[p * E + tid];
            a.psum_chunk[(size_t)blockIdx.x * E + tid] = acc;
        }
    }

    // the last block to arrive finishes the device-wide part
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(a.scan_done, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // counts and per-chunk bases: exclusive scan over chunks, per expert
    int my_count = 0, my_kept = 0;
    if (tid < E) {
        int run = 0;
        int c = 0;
        for (; c + 8 <= a.nchunks; c += 8) {  // 8 independent loads in flight, summed in order
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(&a.chunk_hist[(size_t)(c + u) * E + tid]);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                a.chunk_base[(size_t)(c + u) * E + tid] = run;
                run += v[u];
            }
        }
        for (; c < a.nchunks; ++c) {
            const int v = __ldcg(&a.chunk_hist[(size_t)c * E + tid]);
            a.chunk_base[(size_t)c * E + tid] = run;
            run += v;
        }
        my_count = run;
        my_kept = (a.C < 0) ? run : min(run, a.C);
        a.counts[tid] = my_count;
        a.kept[tid] = my_kept;
    }

    // segment offsets (padded to the GEMM tile), unpadded offsets, M-tile offsets
    const int tiles = ceil_div(my_kept, kSegRows);
    const int v3[3] = {tiles * kSegRows, my_kept, tiles};
    int ex[3], tot[3];
    block_exclusive_scan3(v3, ex, tot, wsum);
    if (tid < E) {
        a.row_off[tid] = ex[0];
        a.kept_off[tid] = ex[1];
        a.mtile_off[tid] = ex[2];
    }
    if (tid == 0) a.mtile_off[E] = tot[2];

    // balance statistic, second level: E * sum_e (counts_e / (T k)) * P_e, P_e the mean
    // router probability, from the scan blocks' partial sums (fixed order)
    if (a.n_router_blocks > 0 && a.aux != nullptr) {
        float* s_part = reinterpret_cast<float*>(sm);
        const int nb = gridDim.x;
        if (tid < P * E) {
            const int ee = tid % E, p = tid / E;
            float acc = 0.0f;
            int q = p;
            for (; q + 3 * P < nb; q += 4 * P) {
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = __ldcg(&a.psum_chunk[(size_t)(q + u * P) * E + ee]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc += v[u];
            }
            for (; q < nb; q += P) acc += __ldcg(&a.psum_chunk[(size_t)q * E + ee]);
            s_part[p * E + ee] = acc;
        }
        __syncthreads();
        double term = 0.0;
        if (tid < E) {
            float Pe = 0.0f;
            for (int p = 0; p < P; ++p) Pe += s_part[p * E + tid];
            term = ((double)my_count / ((double)a.T * (double)a.k)) * ((double)Pe / (double)a.T);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
        if (lane == 0) dsum[warp] = term;
        __syncthreads();
        if (warp == 0) {
            double w = dsum[lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (lane == 0) *a.aux = (float)((double)E * w);
        }
    }

    // the fused expert kernel that follows starts from zeroed scheduler counters
    if (a.ffn_sync != nullptr)
        for (int i = tid; i < a.ffn_sync_n; i += 1024) a.ffn_sync[i] = 0u;
    if (tid == 0) *a.scan_done = 0u;  // re-arm for the next call
}


__global__ void __launch_bounds__(256) k_permute(DispatchArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const long long n_slots = (long long)a.T * a.k;
    const int nvec = a.row_bytes / 16;
    for (long long s = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); s < n_slots;
         s += (long long)gridDim.x * 8) {
        const int t = (int)(s / a.k);
        const int e = a.idx[s];
        const bool e_ok = e >= 0 && e < a.E;
        const int c = (int)(s / kScanChunk);
        const int pos = e_ok ? a.chunk_base[(size_t)c * a.E + e] + a.local_rank[s] : 0;
        const bool keep = e_ok && (a.C < 0 || pos < a.C);
        const int row = keep ? a.row_off[e] + pos : -1;
        if (lane == 0) {
            a.dropped[s] = keep ? 0 : 1;
            if (a.perm_row) a.perm_row[s] = keep ? a.kept_off[e] + pos : -1;
            a.slot_row[s] = row;
            if (keep && a.row_token) {
                a.row_token[row] = t;
                a.row_gate[row] = a.gates[s];
            }
        }
        // top-1 direct combine: a dropped token's output is its input (0 + x = x)
        if (!keep && a.y_pass == nullptr) continue;
        const uint4* src =
            reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)t * a.row_bytes);
        uint4* dst = keep ? reinterpret_cast<uint4*>(static_cast<char*>(a.xp) + (size_t)row * a.row_bytes)
                          : reinterpret_cast<uint4*>(static_cast<char*>(a.y_pass) + (size_t)t * a.row_bytes);
        // up to four 16-byte vectors per lane in flight before any store
        for (int v = lane; v < nvec; v += 128) {
            uint4 r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < nvec) r[u] = ld_stream(src + v + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < nvec) dst[v + 32 * u] = r[u];
        }
    }
}

}  // namespace

size_t dispatch_scan_smem(int E) { return sizeof(int32_t) * 32 * (size_t)(E < 64 ? 64 : E); }

cudaError_t launch_dispatch(const DispatchArgs& a, int num_sms, cudaStream_t st, bool pdl)
{
    const size_t smem = dispatch_scan_smem(a.E);
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k_dispatch_scan), smem);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_kernel(k_dispatch_scan, dim3(a.nchunks), dim3(1024), smem, st, pdl, a);
    if (e != cudaSuccess) return e;
    const long long n_slots = (long long)a.T * a.k;
    long long grid = (n_slots + 7) / 8;
    if (grid > (long long)num_sms * 32) grid = (long long)num_sms * 32;
    return launch_kernel(k_permute, dim3((int)grid), dim3(256), 0, st, true, a);
}

cudaError_t launch_dispatch_scan_only(const DispatchArgs& a, cudaStream_t st)
{
    const size_t smem = dispatch_scan_smem(a.E);
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k_dispatch_scan), smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(k_dispatch_scan, dim3(a.nchunks), dim3(1024), smem, st, false, a);
}

}  // namespace moe
