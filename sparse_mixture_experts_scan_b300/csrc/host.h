// host.h -- host-side pieces shared by the C-ABI files (api.cu, ep.cu): the
// workspace layout of one layer, the per-call context, the validation and the
// four stage launchers.  Internal; not part of the C ABI.
#pragma once

#include <cudaTypedefs.h>

#include "kernels.h"
#include "moe.h"

namespace moe {
namespace host {

constexpr size_t kRegionAlign = 1024;

struct Layout {
    int T, d, F, E, S, k;
    int C;             // capacity, -1 = none
    int n_rblk;        // router blocks
    int nchunks;       // dispatch-scan blocks
    int rows_cap;      // rows of the permuted buffers (multiple of 128)
    int t_pad;         // T rounded up to 128 (shared-expert buffers)
    size_t esz;        // element size of the activation dtype
    bool tc_router;    // bf16 router logits on the tensor core
    bool tc_rbwd;      // router gradients on the tensor core (bf16 layers)
    int r_bn, r_tiles, e_pad;  // router GEMM: MMA N, expert tiles, padded experts
    int r_ksplits;             // router GEMM K splits
    bool r_fuse;               // top-k in the router GEMM's epilogue
    size_t off_wsplit, off_logits;
    size_t off_nsplit, off_nlogits;  // noisy gating: W_noise splits, noise logits [ks, T, E]
    size_t off_psum_chunk;
    size_t off_ffn_sync;  // fused experts: [0] tile counter, [1] finished CTAs, [2..] per-M-tile counts
    int ffn_sync_n;
    size_t off_psum, off_hist, off_base, off_rank, off_slot_row, off_kept, off_row_off,
        off_kept_off, off_mtile, off_xp, off_h, off_yp, off_hs, off_ys;
    size_t off_row_token, off_row_gate;  // token and gate of each permuted row (top-1 direct combine)
    // backward (MOE_FLAG_TRAINING): gate and router gradients, the router's share of dx,
    // dYp (reused for dXp), pre-activations (overwritten in place by their gradients;
    // relu: dZ1 only), shared-expert pre-activations and input gradient
    size_t off_bw_dgate, off_bw_dl, off_bw_dn, off_bw_dxr, off_bw_dyp, off_bw_z1, off_bw_z3, off_bw_zs1,
        off_bw_zs3, off_bw_dxs;
    // router gradients on the tensor core: split gradients, paired weights, dW partials
    int e8, r_nblk, r_dw_splits;
    size_t off_bw_dcat, off_bw_wcat, off_bw_p;
    size_t total;
};

struct Ctx {
    moe_params_t p;
    const moe_inputs_t* in;
    moe_outputs_t* out;
    char* ws;
    Layout L;
    cudaStream_t st;
    int sms;
    bool bf16, use_tc, fused;
    bool pdl = false;  // false until this call has launched its first kernel
    int bn1, bn2;  // MMA N of GEMM1 / GEMM2 (tcgen05 path)
    CUtensorMap mA1, mB1, mB3, mA2, mB2, mAs1, mAs2, mX, mW, mWn;
    CUtensorMap mA1p, mA2p, mAs1p, mAs2p;  // the A maps with kABoxRows-row boxes (partial M-tiles)
    bool q8 = false;              // int8 expert weights
    CUtensorMap mQ1, mQ3, mQ2;    // their uint8 maps
    bool routed_experts = true;   // stage_gemm runs the routed experts (false: shared experts only)
    bool direct_y = false;        // top-1 layer: the fused kernel's GEMM2 epilogue writes y itself
                                  // (and the dispatch copies dropped tokens), no combine launch
    bool wq = false;              // quantised weights on the tensor-memory kernel (k_grouped_gemm_wq)
    int wq_bits = 8, wq_nt = 128; // its weight bits and token rows per tile
    template <typename T>
    T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
    uint32_t* err_word = nullptr;  // where bounded waits report (nullptr: the workspace's first word)
    uint32_t* err() const { return err_word ? err_word : reinterpret_cast<uint32_t*>(ws); }
    unsigned* scan_done() const { return reinterpret_cast<unsigned*>(ws) + 1; }
};

long long capacity_of(const moe_params_t& p);
moe_status_t validate_params(const moe_params_t* p);
Layout make_layout(const moe_params_t& p);
moe_status_t validate_io(const moe_params_t& p, const moe_inputs_t* in, const moe_outputs_t* out);
int sm_count();
// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box {64, box_rows},
// 128-byte swizzle, zero fill out of bounds.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// PDL for every launch of a C-ABI call except its first one.
bool take_pdl(Ctx& c);
// Validates the call, lays out the workspace and encodes the tensor maps.
// io_checked: the inputs and outputs are slices (token ranges) of arrays that
// validate_io already accepted for the whole batch -- their token-indexed [T, k]
// and [T, E] arrays may then start off a 16-byte boundary, which is fine because
// every kernel reads and writes those element by element (the [T, E] logit rows
// are written as 16-byte vectors only when E is a multiple of 4, where a slice
// stays aligned).
moe_status_t prepare(const moe_params_t* params, const moe_inputs_t* in, moe_outputs_t* out, void* ws,
                     size_t ws_bytes, void* stream, Ctx& c, bool io_checked = false);
moe_status_t cuda_status(cudaError_t e);
moe_status_t stage_router(Ctx& c);
moe_status_t stage_dispatch(Ctx& c);
moe_status_t stage_gemm(Ctx& c);
moe_status_t stage_combine(Ctx& c);

}  // namespace host
}  // namespace moe
