// kernels.h -- internal launch interface between the host API (api.cu) and the
// device kernels.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Every launch function takes `pdl`: true lets the launch overlap the tail of the
// previous kernel of the stream (programmatic dependent launch; see common.cuh).
// It is false for the first kernel of each C-ABI call.

// ---- stage 1: router -------------------------------------------------------
struct RouterArgs {
    const void* x;        // [T, d] fp32 or bf16
    const float* Wg;      // [E, d]
    const float* bg;      // [E] or nullptr
    int T, d, E, k, renormalize;
    int32_t* idx;         // [T, k]
    float* gates;         // [T, k]
    float* logits;        // [T, E] or nullptr
    float* probs;         // [T, E] or nullptr
    float* psum_part;     // [router_blocks(T) or router_topk_blocks(T), E] per-block column sums of p
    unsigned* scan_done;  // dispatch-scan arrival counter, reset here
    const float* logit_parts;  // k_router_topk with split-K logits: [k_splits, T, E], else nullptr
    int k_splits;
    // noisy top-k gating (eps == nullptr: off): logits += eps * (softplus(noise + bn) + min_std),
    // noise = the sum of noise_parts[0..k_splits) ([k_splits, T, E], without bn)
    const float* noise_parts;
    const float* bn;      // [E] or nullptr
    const float* eps;     // [T, E] standard normal draws
    float min_std;
    float* raw_out;       // k_router only: write x W^T (no bias, no routing) here and stop
};
// Rows of per-block column sums of p: k_router and the fused tensor-core router write
// one per 32 tokens (router_blocks), k_router_topk one per kTopkTokens tokens.
int router_blocks(int T);
constexpr int kTopkTokens = 8;
int router_topk_blocks(int T);
// CUDA-core router: fp32 logits by FFMA, then softmax / top-k / gates.
cudaError_t launch_router(const RouterArgs& a, bool bf16, cudaStream_t st, bool pdl);
// Softmax / top-k / gates of logits already in a.logits.
cudaError_t launch_router_topk(const RouterArgs& a, cudaStream_t st);


// Tensor-core router logits (bf16 x, W_gate split into three bf16 terms).
struct RouterGemmArgs {
    int T, d, E;
    int E_pad;            // n_tiles * BN rows per split
    int n_tiles;          // expert tiles of BN columns
    int k_splits;         // K split into this many ranges (1: logits + bias written directly)
    const float* bg;      // [E] or nullptr (added here only when k_splits == 1)
    float* logits;        // [T, E] fp32 when k_splits == 1, else [k_splits, T, E] partial sums
    uint32_t* err;
    // fuse != 0 (one tile of at most 32 experts, no K split): softmax, top-k, gates and the
    // per-32-token column sums of p are computed in the epilogue (no separate top-k kernel)
    int fuse, k, renormalize;
    int32_t* idx;         // [T, k]
    float* gates;         // [T, k]
    float* probs;         // [T, E] or nullptr
    float* psum_part;     // [ceil(T / 32), E]
    unsigned* scan_done;  // dispatch-scan arrival counter, reset here
};
int router_tc_bn(int T, int E);  // experts per router GEMM tile (16..64; MMA N = 3x), ~128 CTAs
int router_tc_ksplits(int T, int E, int d);  // K splits so that small batches still fill ~128 CTAs
// The three-term split of an [E, d] fp32 router weight, [router_split_rows(E) / 16][3][16][d]
// bf16 (E rounded up to 64; rows >= E zero): independent of the batch size.
int router_split_rows(int E);
cudaError_t launch_split_wgate(const float* Wg, int E, int d, void* out, int sms, cudaStream_t st, bool pdl);
cudaError_t launch_router_logits_tc(const CUtensorMap& x, const CUtensorMap& w, const RouterGemmArgs& a,
                                    int bn, int sms, cudaStream_t st, bool pdl);

// ---- stage 2: dispatch -----------------------------------------------------
struct DispatchArgs {
    const int32_t* idx;   // [T, k]
    const float* gates;   // [T, k]
    int T, k, E;
    int C;                // capacity, -1 = none
    int nchunks;          // ceil(T*k / kScanChunk)
    int n_router_blocks;
    const float* psum_part;
    float* psum_chunk;    // [nchunks, E] partial sums of psum_part, one row per scan block
    int32_t* local_rank;  // [T*k] rank of the slot among its chunk's slots of the same expert
    int32_t* chunk_hist;  // [nchunks, E]
    int32_t* chunk_base;  // [nchunks, E] exclusive prefix over chunks
    unsigned* scan_done;
    int32_t* counts;      // [E] (user output)
    int32_t* kept;        // [E]
    int32_t* row_off;     // [E] padded segment start rows
    int32_t* kept_off;    // [E] unpadded start rows
    int32_t* mtile_off;   // [E+1]
    float* aux;           // [1] (user output)
    // permute
    const void* x;        // [T, d]
    void* xp;             // [rows_cap, d]
    int row_bytes;        // d * element size
    uint8_t* dropped;     // [T, k]
    int32_t* perm_row;    // [T, k] or nullptr
    int32_t* slot_row;    // [T, k] padded row of the slot or -1
    unsigned* ffn_sync;   // fused-FFN scheduler words cleared by the scan, or nullptr
    int ffn_sync_n;
    // top-1 direct combine (or nullptr): the token and gate of each kept row, and y, into
    // which the permute copies the x row of every dropped token
    int32_t* row_token;
    float* row_gate;
    void* y_pass;
};
size_t dispatch_scan_smem(int E);
cudaError_t launch_dispatch(const DispatchArgs& a, int num_sms, cudaStream_t st, bool pdl);
// The scan kernel alone (no permute); used by the allocation-free entry point.
cudaError_t launch_dispatch_scan_only(const DispatchArgs& a, cudaStream_t st);

// ---- stage 3: grouped GEMMs ------------------------------------------------
// k_ffn_fused_tc loads the token rows (A operand) of a full 128-row M-tile as one box;
// with FusedFfnArgs::partial_a, those of a partial M-tile as the boxes of kABoxRows rows
// that hold valid rows (an expert's last M-tile is mostly padding when it holds few rows,
// and the padding rows were never written): its maps 7-10 are the A maps 0, 3, 5, 6 with
// such boxes.
constexpr int kABoxRows = 32;
// tcgen05 kernel: act is kActNone (plain GEMM), kActRelu, kActGeluTanh,
// kActGeluErf (bias allowed) or kActSwiglu (gated: B rows from W1 and W3).
cudaError_t launch_gemm_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                           const GroupedGemmArgs& args, int act, int bn, int grid,
                           cudaStream_t st, bool pdl);
size_t gemm_tc_smem(int bn);
// Both expert layers of the routed experts in one persistent launch (dynamic tile
// scheduler, GEMM2 tiles wait for the GEMM1 tiles of their M-tile).
struct FusedFfnArgs {
    const int* mtile_off;  // [G+1]
    const int* row_off;    // [G]
    const int* rows;       // [G]
    int G;
    int N1, n_tiles1, K1;  // GEMM1: output columns (d_ff), tiles, reduction (d_model)
    int N2, n_tiles2, K2;  // GEMM2: output columns (d_model), tiles, reduction (d_ff)
    int b1_rows_per_group; // d_ff
    int b2_rows_per_group; // d_model
    void* h;
    int ldh;
    void* yp;
    int ldy;
    const void* bias1;
    const void* bias2;
    void* z1;              // training: GEMM1 pre-activations (W1 half, + bias), [rows, ldh], or nullptr
    void* z3;              // training, SwiGLU: the W3 half
    unsigned* tile_ctr;    // tiles claimed so far (0 at launch)
    unsigned* ctas_done;   // CTAs finished (0 at launch)
    unsigned* mt_done;     // [mt_max] epilogue-warp arrivals per M-tile (0 at launch)
    int mt_max;
    uint32_t* err;
    // Shared experts in the same tile list (S > 0; SwiGLU, no bias): one group of
    // shared_rows token rows read straight from x, hidden S * d_ff (the S experts'
    // W1 / W3 rows are consecutive), GEMM2 over K = S * d_ff in segments of seg_k2
    // columns, segment s reading W2 group b2_group0 + s.  Their GEMM1 tiles come first
    // in the list, their GEMM2 tiles last.
    int S;
    int shared_rows;       // T
    int mt_s;              // M-tiles of the shared group
    int n_tiles_s1;        // GEMM1 column tiles of the shared hidden layer
    int b1_row0;           // first W1 / W3 row of the shared experts (E * d_ff)
    int b2_group0;         // first W2 group of the shared experts (E)
    int seg_k2;            // d_ff, a multiple of 64
    void* hs;              // [T_pad, S * d_ff]
    int ldhs;
    void* ys;              // [T_pad, d_model]
    void* zs1;             // training: the shared pre-activations [T, S * d_ff], or nullptr
    void* zs3;
    int mt_s0;             // first mt_done counter of the shared M-tiles
    // top-1 direct combine (y != nullptr): the GEMM2 epilogue writes
    // y[row_token[r]] = gate * bf16(Yp row r) instead of Yp (ld = ldy)
    void* y;
    const int32_t* row_token;
    const float* row_gate;
    // nonzero: a partial M-tile loads only the kABoxRows-row A boxes that hold valid rows
    // (maps 7-10); zero: every M-tile is one 128-row box
    int partial_a;
};
// maps (11): A1 (Xp), B1 (W1), B3 (W3 or W1), A2 (H), B2 (W2), As1 (x), As2 (Hs), then
// A1, A2, As1, As2 again with kABoxRows-row boxes (the A maps have 128-row boxes); the
// shared-expert maps 5, 6, 9, 10 are read only when S > 0.  MMA N = 256.
cudaError_t launch_ffn_fused_tc(const CUtensorMap* maps, const FusedFfnArgs& a, int act1, int grid,
                                cudaStream_t st, bool pdl);

// int8 expert weights (bf16 activations): tcgen05 grouped GEMM with the int8 B tile
// converted to bf16 in shared memory and the per-output-row scales applied in the
// epilogue.  maps: A (bf16, box {64, 128}), Q and Q3 (uint8 [groups * rows, K], box
// {64, 256} or {64, 128} for the two SwiGLU halves).
struct GroupedGemmQ8Args {
    const int* mtile_off;  // [G+1]
    const int* row_off;    // [G]
    const int* rows;       // [G]
    int G;
    int N, n_tiles, K;
    int b_rows_per_group;  // weight rows (and scales) per group
    void* out;
    int ldo;
    const void* bias;      // [G, b_rows_per_group] bf16 or nullptr
    const float* scale;    // [G, b_rows_per_group] (W1 or W2 rows)
    const float* scale3;   // SwiGLU: the W3 rows' scales
    uint32_t* err;
};
cudaError_t launch_gemm_q8(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& q3,
                           const GroupedGemmQ8Args& args, int act, int grid, cudaStream_t st, bool pdl);
size_t gemm_q8_smem();
// Per-row symmetric int8 quantisation (scale = max|w| / 127, q = rint(w / scale)).
cudaError_t launch_quantize_int8(const void* w, bool bf16, long long rows, int cols, int8_t* q, float* scale,
                                 int sms, cudaStream_t st);

// Quantised expert weights for layers whose experts hold few tokens (the expert
// stage streams the weights): the transposed product D[n, m] = W[n, :] . X[m, :]
// with the weight tile converted to bf16 into tensor memory (the MMA's A operand)
// and the token tile (NT rows) as B.  8-bit: per-row scales applied in the
// epilogue; 4-bit: group scales (128 input columns) applied by the converters (in
// bf16: bf16(q * bf16(scale))).
// maps: X (bf16 [rows, K], box {64, NT}), W and W3 (uint8 [groups * rows, K bytes],
// box {128 bytes, 128 rows}, 128-byte swizzle).
struct GroupedGemmWqArgs {
    const int* row_off;    // [G] padded segment starts of the token rows
    const int* rows;       // [G] token rows per group
    int G;
    int N, n_tiles, K;     // output columns (weight rows per group), gemm_wq_weight_tiles, reduction
    int b_rows_per_group;
    void* out;             // [rows, ldo] bf16
    int ldo;
    const void* bias;      // [G, b_rows_per_group] bf16 or nullptr
    const float* scale;    // 8-bit: [G, b_rows_per_group]; 4-bit: [G, b_rows_per_group, K / 128]
    const float* scale3;   // SwiGLU: the W3 rows' scales
    uint32_t* err;
};
// Token rows per tile (32, 64, 96 or 128; at most 64 for SwiGLU) for a layer whose
// experts hold about rows_per_expert rows.
int gemm_wq_tokens_tile(int rows_per_expert, bool gated);
// Weight-row tiles of an N-row layer: 256 rows (two A tiles) without SwiGLU when
// nt <= 96, else 128 rows.  GroupedGemmWqArgs::n_tiles must be this value.
int gemm_wq_weight_tiles(int N, int act, int nt);
cudaError_t launch_gemm_wq(const CUtensorMap& x, const CUtensorMap& w, const CUtensorMap& w3,
                           const GroupedGemmWqArgs& a, int wbits, int act, int nt, int grid, cudaStream_t st,
                           bool pdl);
// Group-wise symmetric 4-bit quantisation (groups of 128 columns, scale = max|w| / 7,
// q = rint(w / scale) in [-7, 7], two values per byte, low nibble first).
cudaError_t launch_quantize_int4(const void* w, bool bf16, long long rows, int cols, uint8_t* q, float* scale,
                                 int sms, cudaStream_t st);

// FFMA kernel over fp32 or bf16 operands (A [a_rows_alloc, lda], B [*, ldb]).
cudaError_t launch_gemm_ffma(const void* A, int lda, const void* B, const void* B3, int ldb,
                             const GroupedGemmArgs& args, int act, bool bf16, int grid,
                             cudaStream_t st, bool pdl);
constexpr int kFfmaTileN = 64;

// ---- backward: grouped GEMMs ---------------------------------------------------
// C_g[m, n] = sum_k A_g(m, k) B_g(k, n) (+ a second product A2 B2 with the same
// strides), element (m, k) of A at A[a_base + m*a_sm + k*a_sk], (k, n) of B at
// B[b_base + k*b_sk + n*b_sn], output at C[c_base + m*c_sm + n].  Per group g:
//   kBwdRows   M = rows[g]:   a_base = row_off[g]*a_sm, c_base = row_off[g]*c_sm,
//                             b_base = (b_g0+g)*b_gs; tiles from mtile_off (128 rows)
//   kBwdReduce K = rows[g]:   a_base = row_off[g]*a_sk, b_base = row_off[g]*b_sk,
//                             c_base = (c_g0+g)*c_gs; M, N fixed
//   kBwdFixed  one group:     a_base = 0, b_base = b_g0*b_gs, c_base = 0
// Epilogues: store; relu backward (e1 = the saved relu output h); GELU backward
// (e1 = the pre-activation z); SwiGLU backward (e1 = z1, e2 = z3; writes
// dz1 = v z3 silu'(z1) to C and dz3 = v silu(z1) to C2); e1, e2, C2 share C's indexing.
enum BwdMode : int { kBwdFixed = 0, kBwdRows = 1, kBwdReduce = 2 };
enum BwdEpi : int {
    kEpiStore = 0,
    kEpiReluBwd = 1,
    kEpiGeluTanhBwd = 2,
    kEpiGeluErfBwd = 3,
    kEpiSwigluBwd = 4,
    kEpiStoreF32 = 5  // tensor-core kernel only: fp32 output
};
enum BwdTypes : int { kBwdTypesBf16 = 0, kBwdTypesF32 = 1, kBwdTypesF32xBf16 = 2 };  // (A,B,C) element types
struct BwdGemmArgs {
    int mode, epi;
    const void* A;
    const void* A2;
    long long a_sm, a_sk;
    const void* B;
    const void* B2;
    long long b_sk, b_sn, b_gs;
    int b_g0;
    void* C;
    void* C2;
    long long c_sm, c_gs;
    int c_g0;
    const void* e1;
    const void* e2;
    const void* bias;     // store epilogue: + bias[(b_g0 + g) * N + n] (element type of C), or nullptr
    int M, N, K;
    const int* mtile_off;
    const int* row_off;
    const int* rows;
    int G;
};
cudaError_t launch_gemm_bwd_ffma(const BwdGemmArgs& a, int types, int grid, cudaStream_t st, bool pdl);

// tcgen05 version for bf16 (BM = 128, BN = 256, BK = 64).  maps = {A, B, A2, B2}:
//   kBwdRows:   A K-major (box {64, 128}) over the activation-gradient rows; B MN-major
//               (box {64, 64}) over a weight viewed [groups * b_rows_per_group, N-extent];
//               B row of (group g, k) = (b_g0 + g) * b_rows_per_group + k, column b_col0 + n.
//               row_off == nullptr: one group of fixed_rows rows from row 0.
//   kBwdReduce: A and B MN-major (box {64, 64}) over row-major activation buffers; the
//               reduction runs over rows [row_off[g], row_off[g] + rows[g]) (or [0, fixed_rows));
//               output rows m < M of C + (c_g0 + g) * c_gs, leading dimension ldc.
struct BwdTcArgs {
    const int* mtile_off;
    const int* row_off;
    const int* rows;
    int G, fixed_rows;
    int M, N, K;
    int b_g0, b_rows_per_group, b_col0;
    int a_col0;           // kBwdReduce: first A column (M offset)
    int split_rows;       // kBwdReduce with one fixed group: > 0 splits the rows into groups of
                          // this many (group g -> output block c_g0 + g), a split-K over rows;
                          // a multiple of 64 (K blocks never cross into the next group)
    int two_seg;
    void* C;
    void* C2;
    const void* e1;
    const void* e2;
    long long ldc, c_gs;
    int c_g0;
    uint32_t* err;
};
cudaError_t launch_gemm_bwd_tc(const CUtensorMap* maps, const BwdTcArgs& a, int mode, int epi, int grid,
                               cudaStream_t st, bool pdl);

// Zero rows [rows[e], ceil(rows[e] / 64) * 64) of each expert segment in up to three
// row-major buffers (the rows a 64-row K block of a reduction reads past the kept rows).
struct ZeroPadArgs {
    const int* row_off;
    const int* rows;
    int G;
    void* buf[3];
    int row_bytes[3];
};
cudaError_t launch_zero_pad_rows(const ZeroPadArgs& a, int sms, cudaStream_t st, bool pdl);

// Router gradients on the tensor core.  The fp32 logit gradients dl (and dn) are
// split exactly into bf16 terms hi + mid + lo; with E8 = E rounded up to 8:
//   D [T, nblk * E8] = [dl_hi | dl_mid | dl_lo | dl_hi (| the same for dn)]
//   B [nblk * E8, d] = [W_hi; W_hi; W_hi; W_mid (; the same for W_noise)]
// so that D B = dl W_hi + dl_hi W_mid (+ dn ...) ~ dl W_gate (+ dn W_noise), and the
// first three blocks of D reduce against x to three exact-product partials of dW.
cudaError_t launch_split_grad(const float* dl, const float* dn, int T, int E, int E8, int nblk, void* out,
                              int sms, cudaStream_t st, bool pdl);
cudaError_t launch_split_wcat(const float* Wg, const float* Wn, int E, int E8, int d, int nblk, void* out,
                              int sms, cudaStream_t st, bool pdl);
// out[e, i] = sum over splits s (in order) of (P_s[2 E8 + e, i] + P_s[E8 + e, i]) + P_s[e, i], e < E;
// P_s = P + s * 3 E8 d
cudaError_t launch_sum3(const float* P, int splits, int E, int E8, int d, float* out, int sms, cudaStream_t st,
                        bool pdl);
// K splits of the router's dW reduction over T tokens (about one CTA per SM)
int router_dw_splits(int T, int E8, int d);

// ---- backward: memory-bound kernels ---------------------------------------------
struct BwdCombineArgs {
    const void* dy;        // [T, d]
    const void* yp;        // [rows_cap, d] forward expert outputs
    void* dyp;             // [rows_cap, d] out: gate * dy on the slot's row
    const int32_t* slot_row;
    const float* gates;    // [T, k]
    float* dgate;          // [T, k] out
    int T, d, k;
};
cudaError_t launch_bwd_combine(const BwdCombineArgs& a, bool bf16, int sms, cudaStream_t st, bool pdl);

struct RouterBwdArgs {
    const float* logits;   // [T, E] the logits the gating used
    const int32_t* idx;    // [T, k]
    const float* dgate;    // [T, k]
    const int32_t* counts; // [E]
    float d_aux;
    int T, E, k, renormalize;
    float* dl;             // [T, E] out
    // noisy gating (eps == nullptr: off)
    const float* noise_parts;  // [k_splits, T, E] noise logits without b_noise
    int k_splits;
    const float* bn;
    const float* eps;
    float* dn;             // [T, E] out
};
cudaError_t launch_router_bwd(const RouterBwdArgs& a, int sms, cudaStream_t st, bool pdl);

// out[(out_g0 + g) * N + n] = sum_{r < rows[g]} A[(row_off[g] + r) * lda + n]
// (row_off == nullptr: one group of fixed_rows rows from row 0)
struct ColsumArgs {
    const void* A;
    long long lda;
    const int* row_off;
    const int* rows;
    int fixed_rows;
    int G, N, out_g0;
    void* out;
};
cudaError_t launch_colsum(const ColsumArgs& a, int types, int sms, cudaStream_t st, bool pdl);

struct BwdUnpermuteArgs {
    const void* dy;        // [T, d]
    const void* dxp;       // [rows_cap, d]
    const void* dxs;       // [T, d] shared experts' input gradient, or nullptr
    const float* dxr;      // [T, d] router's input gradient
    const int32_t* slot_row;
    int T, d, k, residual_mode;
    void* dx;              // [T, d] out
};
cudaError_t launch_bwd_unpermute(const BwdUnpermuteArgs& a, bool bf16, int sms, cudaStream_t st, bool pdl);

// ---- diagnostics ------------------------------------------------------------
// One kernel whose bounded wait on a barrier nobody arrives at expires after
// timeout_ns and sets an error bit in *err, as the layer's kernels do on expiry.
cudaError_t launch_wait_expires(uint32_t* err, unsigned long long timeout_ns, cudaStream_t st);

// ---- stage 4: combine ------------------------------------------------------
struct CombineArgs {
    const void* yp;       // [rows_cap, d]
    const void* ys;       // [T_pad, d] shared-expert output or nullptr
    const void* x;        // [T, d]
    const int32_t* slot_row;
    const float* gates;
    void* y;              // [T, d]
    int T, k, d, residual_mode;
    int seg_vec;          // 16-byte vectors per work item (set by launch_combine)
};
cudaError_t launch_combine(const CombineArgs& a, bool bf16, int num_sms, cudaStream_t st, bool pdl);

}  // namespace moe
