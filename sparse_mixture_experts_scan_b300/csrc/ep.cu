// ep.cu -- expert parallelism over G virtual ranks on one GPU.
//
// "MoE架构解析" §3.2 (分布式训练优化): the experts are placed on different
// devices and, in the mixed data + expert parallel mode, the data is sharded
// over the workers, each worker holds a part of the experts and tokens travel
// between devices; §5 (问题3) names the exchange, an AllToAll.
// "MoE混合专家模型原理与实战" §4.2 (专家分片): 64 experts cut over 4 cards.
//
// Rank r holds the tokens [floor(r T / G), floor((r+1) T / G)) and the experts
// [r E/G, (r+1) E/G).  Every rank owns a private workspace (the single-rank
// layout of its shard), so the only data that crosses ranks is what the
// exchange kernels below move:
//   1. each rank routes its shard and dispatches it into its send buffer
//      (the single-rank router and dispatch; capacity C_r = floor(T_r cf / E),
//      the pages' rule applied to the shard);
//   2. k_ep_plan: the counts exchange -- every destination learns how many
//      rows each source sends per expert (kept counts of all ranks), lays out
//      its receive buffer (its experts in ascending order, inside one expert
//      the rows of rank 0, 1, ..., each padded segment a multiple of the GEMM
//      tile), and the balance statistic is reduced over all ranks;
//   3. k_ep_send: the token all-to-all, one warp per slot, from the source's
//      send buffer into the owner's receive buffer;
//   4. each destination runs its experts on the rows it received (the fused
//      tcgen05 expert kernel, or the FFMA kernel for fp32 layers);
//   5. k_ep_return: the reverse all-to-all, the expert outputs back into the
//      source's buffer at the rows its dispatch gave them;
//   6. each rank applies the shared experts to its own tokens and combines.
// On one GPU the G ranks are emulated as buffers; all kernels run in order on
// the caller's stream.  No peer memory, NVLink multicast or collective
// library is involved.
#include <algorithm>

#include "host.h"

namespace moe {
namespace {

constexpr int kEpMaxRanks = MOE_EP_MAX_RANKS;

struct EpArgs {
    int G, E, E_loc, T, k, row_bytes;
    int t0[kEpMaxRanks + 1];                // token shard bounds
    const int32_t* kept[kEpMaxRanks];       // [E] rows of each expert in the rank's send buffer
    const int32_t* row_off[kEpMaxRanks];    // [E] their padded segment starts
    const int32_t* slot_row[kEpMaxRanks];   // [T_r k] padded send-buffer row of each slot, -1 dropped
    const float* psum_chunk[kEpMaxRanks];   // [nchunks_r, E] the rank's probability-sum partials
    int nchunks[kEpMaxRanks];
    const char* xp[kEpMaxRanks];            // send buffers (the ranks' permuted token rows)
    char* yp[kEpMaxRanks];                  // return buffers (expert outputs, send-buffer rows)
    char* xr[kEpMaxRanks];                  // receive buffers of the owners
    const char* yr[kEpMaxRanks];            // the owners' expert outputs
    unsigned* ffn_sync[kEpMaxRanks];        // the owners' fused-kernel scheduler words
    int sync_n;
    const int32_t* counts_rank;             // [G, E] pre-drop counts of each rank's tokens
    const int32_t* idx;                     // [T, k] selected experts (all ranks)
    int32_t* base;                          // [G, E] rows of expert e sent by ranks < r
    int32_t* tot;                           // [E] rows of expert e over all ranks
    int32_t* gkept_off;                     // [E] unpadded start of expert e in the concatenation
    int32_t* recv_row_off;                  // [E] padded start of expert e in its owner's buffer
    int32_t* recv_mtile;                    // [G, E_loc + 1] M-tile offsets of each owner
    int32_t* recv_slot_row;                 // [T k] padded receive row of each slot, -1 dropped
    int32_t* counts;                        // [E] output: all ranks' counts
    float* aux;                             // [1] output: balance statistic over all ranks
    int32_t* perm_row;                      // [T k] output or nullptr
};

__device__ __forceinline__ int rank_of(const EpArgs& a, int t)
{
    int r = 0;
    while (r + 1 < a.G && t >= a.t0[r + 1]) ++r;
    return r;
}

// Exclusive scan of three ints over the block's 1024 threads, in thread order.
__device__ void ep_block_scan3(const int (&v)[3], int (&out)[3], int (*wsum)[3])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int u = __shfl_up_sync(0xffffffffu, inc[q], o);
            if (lane >= o) inc[q] += u;
        }
    if (lane == 31)
#pragma unroll
        for (int q = 0; q < 3; ++q) wsum[warp][q] = inc[q];
    __syncthreads();
    if (warp == 0)
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
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) out[q] = (warp > 0 ? wsum[warp - 1][q] : 0) + inc[q] - v[q];
    __syncthreads();
}

// The counts exchange and the receive layouts (one block; thread e = expert e).
__global__ void __launch_bounds__(1024) k_ep_plan(EpArgs a)
{
    __shared__ int wsum[32][3];
    __shared__ int s_pad[kMaxExperts], s_mt[kMaxExperts];
    __shared__ double dsum[32];
    __shared__ float s_part[1024];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, E = a.E;
    // probability sums: thread (e, p) adds the rows p, p + Pn, ... of every rank's
    // partials of expert e (loads issued four at a time); the Pn slices are then added
    // in a fixed order
    const int Pn = 1024 / E;
    if (tid < Pn * E) {
        const int e = tid % E, p = tid / E;
        float acc = 0.0f;
        for (int r = 0; r < a.G; ++r) {
            if (a.t0[r + 1] <= a.t0[r]) continue;  // an empty shard ran no dispatch
            const float* src = a.psum_chunk[r];
            const int nc = a.nchunks[r];
            int c = p;
            for (; c + 3 * Pn < nc; c += 4 * Pn) {
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = __ldcg(&src[(size_t)(c + u * Pn) * E + e]);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc += v[u];
            }
            for (; c < nc; c += Pn) acc += __ldcg(&src[(size_t)c * E + e]);
        }
        s_part[tid] = acc;
    }
    // kept and pre-drop counts of every rank (independent loads first)
    int kk[kEpMaxRanks], cc[kEpMaxRanks];
    int tot = 0, cnt = 0;
    float P = 0.0f;
    if (tid < E) {
#pragma unroll
        for (int r = 0; r < kEpMaxRanks; ++r) {
            const bool has = r < a.G && a.t0[r + 1] > a.t0[r];
            kk[r] = has ? __ldcg(&a.kept[r][tid]) : 0;
            cc[r] = has ? __ldcg(&a.counts_rank[r * E + tid]) : 0;
        }
#pragma unroll
        for (int r = 0; r < kEpMaxRanks; ++r) {
            if (r < a.G) a.base[r * E + tid] = tot;
            tot += kk[r];
            cnt += cc[r];
        }
        a.tot[tid] = tot;
        a.counts[tid] = cnt;
    }
    __syncthreads();
    if (tid < E)
        for (int p = 0; p < Pn; ++p) P += s_part[p * E + tid];
    const int tiles = ceil_div(tot, kSegRows);
    const int v3[3] = {tiles * kSegRows, tot, tiles};
    int ex[3];
    ep_block_scan3(v3, ex, wsum);
    if (tid < E) {
        s_pad[tid] = ex[0];
        s_mt[tid] = ex[2];
        a.gkept_off[tid] = ex[1];
    }
    __syncthreads();
    if (tid < E) {
        const int q = tid / a.E_loc, first = q * a.E_loc, el = tid - first;
        a.recv_row_off[tid] = ex[0] - s_pad[first];
        a.recv_mtile[q * (a.E_loc + 1) + el] = ex[2] - s_mt[first];
        if (el == a.E_loc - 1) a.recv_mtile[q * (a.E_loc + 1) + a.E_loc] = ex[2] + tiles - s_mt[first];
    }
    // E * sum_e (counts_e / (T k)) * (P_e / T) over every rank's tokens
    double term = 0.0;
    if (tid < E) term = ((double)cnt / ((double)a.T * (double)a.k)) * ((double)P / (double)a.T);
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
    // the owners' fused expert kernels start from zeroed scheduler words
    for (int q = 0; q < a.G; ++q)
        if (a.ffn_sync[q] != nullptr)
            for (int i = tid; i < a.sync_n; i += 1024) a.ffn_sync[q][i] = 0u;
}

// Copy one row of row_bytes bytes with the lanes of a warp (16-byte vectors,
// up to four in flight per lane before the stores).
__device__ __forceinline__ void copy_row(const char* src, char* dst, int row_bytes, int lane)
{
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int nvec = row_bytes / 16;
    for (int v = lane; v < nvec; v += 128) {
        uint4 r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v + 32 * u < nvec) r[u] = ld_stream(s + v + 32 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v + 32 * u < nvec) d[v + 32 * u] = r[u];
    }
}

// The token all-to-all: every kept slot's row goes from its rank's send buffer
// to the receive buffer of its expert's owner.  One warp per slot.
__global__ void __launch_bounds__(256) k_ep_send(EpArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const long long n_slots = (long long)a.T * a.k;
    for (long long s = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); s < n_slots;
         s += (long long)gridDim.x * 8) {
        const int t = (int)(s / a.k);
        const int r = rank_of(a, t);
        const long long s_loc = s - (long long)a.t0[r] * a.k;
        const int src_row = a.slot_row[r][s_loc];
        const int e = a.idx[s];
        if (src_row < 0 || e < 0 || e >= a.E) {
            if (lane == 0) {
                a.recv_slot_row[s] = -1;
                if (a.perm_row) a.perm_row[s] = -1;
            }
            continue;
        }
        const int pos = src_row - a.row_off[r][e];
        const int q = e / a.E_loc;
        const int before = a.base[r * a.E + e];
        const int dst_row = a.recv_row_off[e] + before + pos;
        if (lane == 0) {
            a.recv_slot_row[s] = dst_row;
            if (a.perm_row) a.perm_row[s] = a.gkept_off[e] + before + pos;
        }
        copy_row(a.xp[r] + (size_t)src_row * a.row_bytes, a.xr[q] + (size_t)dst_row * a.row_bytes, a.row_bytes,
                 lane);
    }
}

// The reverse all-to-all: each kept slot's expert output goes back to its
// rank's buffer, at the row the rank's dispatch gave the slot.
__global__ void __launch_bounds__(256) k_ep_return(EpArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const long long n_slots = (long long)a.T * a.k;
    for (long long s = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); s < n_slots;
         s += (long long)gridDim.x * 8) {
        const int dst_row = a.recv_slot_row[s];
        if (dst_row < 0) continue;
        const int t = (int)(s / a.k);
        const int r = rank_of(a, t);
        const int src_row = a.slot_row[r][s - (long long)a.t0[r] * a.k];
        const int q = a.idx[s] / a.E_loc;
        copy_row(a.yr[q] + (size_t)dst_row * a.row_bytes, a.yp[r] + (size_t)src_row * a.row_bytes, a.row_bytes,
                 lane);
    }
}

// ---------------------------------------------------------------------------
// host side

constexpr size_t kAlign = 1024;

struct EpPlan {
    int G, E_loc;
    int t0[kEpMaxRanks + 1];
    moe_params_t pr[kEpMaxRanks];
    size_t off_ws[kEpMaxRanks], ws_bytes[kEpMaxRanks];
    size_t off_cnt, off_auxr, off_base, off_tot, off_gkept, off_rrow, off_rmt, off_rslot;
    int rows_recv, sync_n;
    size_t off_xr[kEpMaxRanks], off_h[kEpMaxRanks], off_yr[kEpMaxRanks], off_sync[kEpMaxRanks];
    size_t total;
};

moe_status_t ep_validate(const moe_params_t* p, int G)
{
    moe_status_t s = host::validate_params(p);
    if (s != MOE_OK) return s;
    if (G < 1 || G > kEpMaxRanks || p->E % G != 0) return MOE_ERR_INVALID_ARG;
    // the exchange feeds the single-launch expert kernels of the owners: the fused
    // tcgen05 kernel (bf16) or the FFMA kernel (fp32, or bf16 with MOE_FLAG_FFMA_EXPERTS);
    // int8 weights, the two-launch cross-check path and the backward are not built here
    if (p->weight_format != MOE_WEIGHTS_DTYPE || (p->flags & (MOE_FLAG_UNFUSED_EXPERTS | MOE_FLAG_TRAINING)))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

EpPlan ep_plan(const moe_params_t& p, int G)
{
    EpPlan P{};
    P.G = G;
    P.E_loc = p.E / G;
    for (int r = 0; r <= G; ++r) P.t0[r] = (int)((long long)r * p.T / G);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + kAlign - 1) / kAlign * kAlign;
        return at;
    };
    long long cap_sum = 0;  // sum over ranks of the per-shard capacity (-1: no limit)
    bool capped = true;
    for (int r = 0; r < G; ++r) {
        P.pr[r] = p;
        P.pr[r].T = P.t0[r + 1] - P.t0[r];
        P.ws_bytes[r] = host::make_layout(P.pr[r]).total;
        P.off_ws[r] = take(P.ws_bytes[r]);
        const long long C = host::capacity_of(P.pr[r]);
        if (C < 0) capped = false;
        else cap_sum += C;
    }
    const size_t E = (size_t)p.E;
    const long long slots = (long long)p.T * p.k;
    P.off_cnt = take(sizeof(int32_t) * G * E);
    P.off_auxr = take(sizeof(float) * G);
    P.off_base = take(sizeof(int32_t) * G * E);
    P.off_tot = take(sizeof(int32_t) * E);
    P.off_gkept = take(sizeof(int32_t) * E);
    P.off_rrow = take(sizeof(int32_t) * E);
    P.off_rmt = take(sizeof(int32_t) * G * (P.E_loc + 1));
    P.off_rslot = take(sizeof(int32_t) * (size_t)std::max(slots, 1ll));
    // an owner receives at most every slot (or every shard's capacity for each of
    // its experts), plus the padding of its expert segments to the GEMM tile
    long long recv = slots;
    if (capped) recv = std::min(recv, (long long)P.E_loc * cap_sum);
    recv += (long long)P.E_loc * (kSegRows - 1);
    if (capped) recv = std::min(recv, (long long)P.E_loc * ((cap_sum + kSegRows - 1) / kSegRows * kSegRows));
    P.rows_recv = (int)((recv + kSegRows - 1) / kSegRows * kSegRows);
    P.sync_n = 2 + P.rows_recv / kSegRows;
    const size_t esz = p.dtype == MOE_BF16 ? 2 : 4;
    for (int q = 0; q < G; ++q) {
        P.off_xr[q] = take(esz * (size_t)P.rows_recv * p.d_model);
        P.off_h[q] = take(esz * (size_t)P.rows_recv * p.d_ff);
        P.off_yr[q] = take(esz * (size_t)P.rows_recv * p.d_model);
        P.off_sync[q] = take(sizeof(unsigned) * P.sync_n);
    }
    P.total = o;
    return P;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

const void* offset_bytes(const void* p, size_t n) { return p ? static_cast<const char*>(p) + n : nullptr; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_ep_workspace_size(const moe_params_t* params, int32_t G, size_t* bytes)
{
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t s = ep_validate(params, G);
    if (s != MOE_OK) return s;
    *bytes = ep_plan(*params, G).total;
    return MOE_OK;
}

extern "C" moe_status_t moe_forward_ep(const moe_params_t* params, int32_t G, const moe_inputs_t* inputs,
                                       moe_outputs_t* outputs, void* workspace, size_t workspace_bytes,
                                       void* stream)
{
    moe_status_t s = ep_validate(params, G);
    if (s != MOE_OK) return s;
    const moe_params_t& p = *params;
    s = host::validate_io(p, inputs, outputs);
    if (s != MOE_OK) return s;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_WORKSPACE;
    const EpPlan P = ep_plan(p, G);
    if (workspace_bytes < P.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.T == 0) {
        cudaError_t e = cudaMemsetAsync(outputs->counts, 0, sizeof(int32_t) * p.E, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(outputs->aux, 0, sizeof(float), st);
        return host::cuda_status(e);
    }
    const size_t esz = p.dtype == MOE_BF16 ? 2 : 4;
    const size_t row_bytes = esz * (size_t)p.d_model;

    // ---- every rank's view of the layer: its token shard, its slices of the
    // outputs and its private workspace
    host::Ctx ctx[kEpMaxRanks];
    moe_inputs_t in_r[kEpMaxRanks];
    moe_outputs_t out_r[kEpMaxRanks];
    for (int r = 0; r < G; ++r) {
        const size_t t0 = (size_t)P.t0[r];
        in_r[r] = *inputs;
        in_r[r].x = offset_bytes(inputs->x, t0 * row_bytes);
        in_r[r].noise_eps = static_cast<const float*>(offset_bytes(inputs->noise_eps, t0 * p.E * sizeof(float)));
        out_r[r] = *outputs;
        out_r[r].y = const_cast<void*>(offset_bytes(outputs->y, t0 * row_bytes));
        out_r[r].expert_idx = outputs->expert_idx + t0 * p.k;
        out_r[r].gates = outputs->gates + t0 * p.k;
        out_r[r].dropped = outputs->dropped + t0 * p.k;
        out_r[r].counts = at<int32_t>(workspace, P.off_cnt) + (size_t)r * p.E;
        out_r[r].aux = at<float>(workspace, P.off_auxr) + r;
        out_r[r].logits = outputs->logits ? outputs->logits + t0 * p.E : nullptr;
        out_r[r].probs = outputs->probs ? outputs->probs + t0 * p.E : nullptr;
        out_r[r].perm_row = nullptr;  // written below, in the concatenated receive order
        s = host::prepare(&P.pr[r], &in_r[r], &out_r[r], at<void>(workspace, P.off_ws[r]), P.ws_bytes[r], stream,
                          ctx[r], /*io_checked=*/true);
        if (s != MOE_OK) return s;
        // every rank's bounded waits report to the first word of the caller's workspace
        ctx[r].err_word = at<uint32_t>(workspace, 0);
        // the owners run the experts here, so every rank combines with k_combine
        ctx[r].direct_y = false;
    }
    // the owners' expert kernels: tensor maps over the receive buffers and the
    // owner's slice of the expert weights
    const bool bf16 = p.dtype == MOE_BF16;
    const bool use_tc = bf16 && !(p.flags & MOE_FLAG_FFMA_EXPERTS);
    const bool gated = p.act == MOE_ACT_SWIGLU;
    const int E_loc = P.E_loc;
    CUtensorMap maps[kEpMaxRanks][11] = {};  // the fused kernel's maps (no shared experts: 5, 6, 9, 10 unused)
    if (use_tc) {
        const int b1_rows = gated ? 128 : 256;
        for (int q = 0; q < G; ++q) {
            const size_t w13 = (size_t)q * E_loc * p.d_ff * p.d_model * esz;
            bool ok = host::encode_bf16_2d(&maps[q][0], at<void>(workspace, P.off_xr[q]), P.rows_recv, p.d_model, 128) &&
                      host::encode_bf16_2d(&maps[q][7], at<void>(workspace, P.off_xr[q]), P.rows_recv, p.d_model,
                                           kABoxRows) &&
                      host::encode_bf16_2d(&maps[q][8], at<void>(workspace, P.off_h[q]), P.rows_recv, p.d_ff,
                                           kABoxRows) &&
                      host::encode_bf16_2d(&maps[q][1], offset_bytes(inputs->W1, w13), (uint64_t)E_loc * p.d_ff,
                                           p.d_model, b1_rows) &&
                      host::encode_bf16_2d(&maps[q][2], offset_bytes(gated ? inputs->W3 : inputs->W1, w13),
                                           (uint64_t)E_loc * p.d_ff, p.d_model, b1_rows) &&
                      host::encode_bf16_2d(&maps[q][3], at<void>(workspace, P.off_h[q]), P.rows_recv, p.d_ff, 128) &&
                      host::encode_bf16_2d(&maps[q][4], offset_bytes(inputs->W2, w13), (uint64_t)E_loc * p.d_model,
                                           p.d_ff, 256);
            if (!ok) return MOE_ERR_UNSUPPORTED;
        }
    }

    EpArgs a{};
    a.G = G;
    a.E = p.E;
    a.E_loc = E_loc;
    a.T = p.T;
    a.k = p.k;
    a.row_bytes = (int)row_bytes;
    for (int r = 0; r <= G; ++r) a.t0[r] = P.t0[r];
    for (int r = 0; r < G; ++r) {
        const host::Ctx& c = ctx[r];
        a.kept[r] = c.at<int32_t>(c.L.off_kept);
        a.row_off[r] = c.at<int32_t>(c.L.off_row_off);
        a.slot_row[r] = c.at<int32_t>(c.L.off_slot_row);
        a.psum_chunk[r] = c.at<float>(c.L.off_psum_chunk);
        a.nchunks[r] = c.L.nchunks;
        a.xp[r] = c.at<char>(c.L.off_xp);
        a.yp[r] = c.at<char>(c.L.off_yp);
        a.xr[r] = at<char>(workspace, P.off_xr[r]);
        a.yr[r] = at<char>(workspace, P.off_yr[r]);
        a.ffn_sync[r] = use_tc ? at<unsigned>(workspace, P.off_sync[r]) : nullptr;
    }
    a.sync_n = P.sync_n;
    a.counts_rank = at<int32_t>(workspace, P.off_cnt);
    a.idx = outputs->expert_idx;
    a.base = at<int32_t>(workspace, P.off_base);
    a.tot = at<int32_t>(workspace, P.off_tot);
    a.gkept_off = at<int32_t>(workspace, P.off_gkept);
    a.recv_row_off = at<int32_t>(workspace, P.off_rrow);
    a.recv_mtile = at<int32_t>(workspace, P.off_rmt);
    a.recv_slot_row = at<int32_t>(workspace, P.off_rslot);
    a.counts = outputs->counts;
    a.aux = outputs->aux;
    a.perm_row = outputs->perm_row;

    // ---- the launch sequence (one stream; every launch after the first overlaps
    // its predecessor's tail by programmatic dependent launch)
    bool pdl = false;
    auto next_pdl = [&] {
        const bool v = pdl;
        pdl = true;
        return v;
    };
    auto sync_pdl = [&](host::Ctx& c) { c.pdl = pdl; };
    auto after = [&](host::Ctx& c) { pdl = pdl || c.pdl; };
    // 1. routing and dispatch into the send buffers, rank by rank
    for (int r = 0; r < G; ++r) {
        sync_pdl(ctx[r]);
        s = host::stage_router(ctx[r]);
        after(ctx[r]);
        if (s != MOE_OK) return s;
    }
    for (int r = 0; r < G; ++r) {
        sync_pdl(ctx[r]);
        s = host::stage_dispatch(ctx[r]);
        after(ctx[r]);
        if (s != MOE_OK) return s;
    }
    const int sms = ctx[0].sms;
    const long long n_slots = (long long)p.T * p.k;
    const int slot_grid = (int)std::min<long long>((n_slots + 7) / 8, (long long)sms * 32);
    // 2. counts exchange and receive layouts, 3. token all-to-all
    cudaError_t e = launch_kernel(k_ep_plan, dim3(1), dim3(1024), 0, st, next_pdl(), a);
    if (e == cudaSuccess) e = launch_kernel(k_ep_send, dim3(slot_grid), dim3(256), 0, st, next_pdl(), a);
    // 4. each owner runs its experts on the rows it received
    const int mt = P.rows_recv / kSegRows;
    for (int q = 0; q < G && e == cudaSuccess; ++q) {
        const int* mtile = at<int>(workspace, P.off_rmt) + q * (E_loc + 1);
        const int* roff = at<int>(workspace, P.off_rrow) + q * E_loc;
        const int* rows = at<int>(workspace, P.off_tot) + q * E_loc;
        if (use_tc) {
            FusedFfnArgs f{};
            f.mtile_off = mtile;
            f.row_off = roff;
            f.rows = rows;
            f.G = E_loc;
            f.N1 = p.d_ff;
            f.n_tiles1 = ceil_div(p.d_ff, gated ? 128 : 256);
            f.K1 = p.d_model;
            f.N2 = p.d_model;
            f.n_tiles2 = ceil_div(p.d_model, 256);
            f.K2 = p.d_ff;
            f.b1_rows_per_group = p.d_ff;
            f.b2_rows_per_group = p.d_model;
            f.h = at<void>(workspace, P.off_h[q]);
            f.ldh = p.d_ff;
            f.yp = at<void>(workspace, P.off_yr[q]);
            f.ldy = p.d_model;
            f.bias1 = offset_bytes(inputs->b1, (size_t)q * E_loc * p.d_ff * esz);
            f.bias2 = offset_bytes(inputs->b2, (size_t)q * E_loc * p.d_model * esz);
            unsigned* sync = at<unsigned>(workspace, P.off_sync[q]);
            f.tile_ctr = sync;
            f.ctas_done = sync + 1;
            f.mt_done = sync + 2;
            f.mt_max = P.sync_n - 2;
            f.err = ctx[q].err();
            // owners whose experts hold about one M-tile each load only the valid rows of
            // a partial M-tile (maps 7 and 8), as the single-rank layer does
            f.partial_a = mt <= E_loc ? 1 : 0;
            const int grid = std::max(1, std::min(mt * (f.n_tiles1 + f.n_tiles2), sms));
            e = launch_ffn_fused_tc(maps[q], f, p.act, grid, st, next_pdl());
        } else {
            GroupedGemmArgs g1{};
            g1.mtile_off = mtile;
            g1.row_off = roff;
            g1.rows = rows;
            g1.G = E_loc;
            g1.N = p.d_ff;
            g1.n_tiles = ceil_div(p.d_ff, kFfmaTileN);
            g1.K = p.d_model;
            g1.k_segments = 1;
            g1.b_rows_per_group = p.d_ff;
            g1.b_group0 = q * E_loc;
            g1.out = at<void>(workspace, P.off_h[q]);
            g1.ldo = p.d_ff;
            g1.bias = inputs->b1;
            g1.a_rows_alloc = P.rows_recv;
            g1.err = ctx[q].err();
            GroupedGemmArgs g2 = g1;
            g2.N = p.d_model;
            g2.n_tiles = ceil_div(p.d_model, kFfmaTileN);
            g2.K = p.d_ff;
            g2.b_rows_per_group = p.d_model;
            g2.out = at<void>(workspace, P.off_yr[q]);
            g2.ldo = p.d_model;
            g2.bias = inputs->b2;
            auto grid_for = [&](int tiles) { return std::max(1, std::min(tiles, sms * 4)); };
            e = launch_gemm_ffma(at<void>(workspace, P.off_xr[q]), p.d_model, inputs->W1, inputs->W3, p.d_model, g1,
                                 p.act, bf16, grid_for(mt * g1.n_tiles), st, next_pdl());
            if (e == cudaSuccess)
                e = launch_gemm_ffma(at<void>(workspace, P.off_h[q]), p.d_ff, inputs->W2, nullptr, p.d_ff, g2,
                                     kActNone, bf16, grid_for(mt * g2.n_tiles), st, next_pdl());
        }
    }
    // 5. the reverse all-to-all
    if (e == cudaSuccess) e = launch_kernel(k_ep_return, dim3(slot_grid), dim3(256), 0, st, next_pdl(), a);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // 6. shared experts on each rank's own tokens, then the combine
    for (int r = 0; r < G; ++r) {
        if (p.n_shared > 0) {
            ctx[r].routed_experts = false;
            sync_pdl(ctx[r]);
            s = host::stage_gemm(ctx[r]);
            after(ctx[r]);
            if (s != MOE_OK) return s;
        }
        sync_pdl(ctx[r]);
        s = host::stage_combine(ctx[r]);
        after(ctx[r]);
        if (s != MOE_OK) return s;
    }
    return MOE_OK;
}
