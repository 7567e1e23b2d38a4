// api.cu -- the C ABI (include/moe.h): validation, workspace layout, TMA tensor
// maps and the launch sequence of the four stages on the caller's stream.
//
// Nothing here allocates device memory or synchronises the host (except
// moe_last_device_status).  Every check happens before the first launch of a
// call, so a non-OK status means nothing was enqueued.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "host.h"

namespace moe {

std::atomic<unsigned long long>& launch_counter()
{
    static std::atomic<unsigned long long> n{0};
    return n;
}

namespace host {

long long capacity_of(const moe_params_t& p)
{
    if (!(p.capacity_factor > 0.0f)) return -1;
    // "MoE架构解析" §3.1: int(batch_size * capacity_factor / num_experts)
    const double c = std::floor((double)p.T * (double)p.capacity_factor / (double)p.E);
    return (long long)std::min(c, (double)p.T);  // C >= T never drops anything
}

moe_status_t validate_params(const moe_params_t* p)
{
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (p->T < 0 || p->d_model < 8 || p->d_ff < 8) return MOE_ERR_INVALID_ARG;
    if (p->d_model % 8 != 0 || p->d_ff % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (p->E < 1 || p->E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
    if (p->k < 1 || p->k > p->E || p->k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (p->n_shared < 0) return MOE_ERR_INVALID_ARG;
    if (p->renormalize != 0 && p->renormalize != 1) return MOE_ERR_INVALID_ARG;
    if (p->residual_mode != 0 && p->residual_mode != 1) return MOE_ERR_INVALID_ARG;
    if (p->act < MOE_ACT_RELU || p->act > MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
    if (p->dtype != MOE_F32 && p->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if ((p->flags & ~(MOE_FLAG_FFMA_EXPERTS | MOE_FLAG_FFMA_ROUTER | MOE_FLAG_UNFUSED_EXPERTS | MOE_FLAG_TRAINING)) !=
        0u)
        return MOE_ERR_INVALID_ARG;
    if (std::isnan(p->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (p->noisy_gating != 0 && p->noisy_gating != 1) return MOE_ERR_INVALID_ARG;
    if (p->weight_format != MOE_WEIGHTS_DTYPE && p->weight_format != MOE_WEIGHTS_INT8 &&
        p->weight_format != MOE_WEIGHTS_INT4)
        return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(p->noise_min_std) || p->noise_min_std < 0.0f) return MOE_ERR_INVALID_ARG;
    if (p->n_shared > 0 && p->act != MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED;
    if (p->weight_format == MOE_WEIGHTS_INT8 &&
        (p->dtype != MOE_BF16 || (p->flags & (MOE_FLAG_FFMA_EXPERTS | MOE_FLAG_TRAINING)) || p->n_shared != 0 ||
         p->d_model % 16 != 0 || p->d_ff % 16 != 0))
        return MOE_ERR_UNSUPPORTED;
    if (p->weight_format == MOE_WEIGHTS_INT4 &&
        (p->dtype != MOE_BF16 || (p->flags & (MOE_FLAG_FFMA_EXPERTS | MOE_FLAG_TRAINING)) || p->n_shared != 0 ||
         p->d_model % MOE_INT4_GROUP != 0 || p->d_ff % MOE_INT4_GROUP != 0))
        return MOE_ERR_UNSUPPORTED;
    // every index and row count below must fit in int32
    const long long slots = (long long)p->T * p->k;
    const long long rows = slots + (long long)p->E * kSegRows + kSegRows;
    const long long t_pad = ((long long)p->T + kSegRows - 1) / kSegRows * kSegRows;
    if (rows >= (1ll << 31) || (long long)(p->E + p->n_shared) * p->d_ff >= (1ll << 31) ||
        (long long)(p->E + p->n_shared) * p->d_model >= (1ll << 31) ||
        (long long)p->n_shared * p->d_ff >= (1ll << 31) || t_pad >= (1ll << 31))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

Layout make_layout(const moe_params_t& p)
{
    Layout L{};
    L.T = p.T;
    L.d = p.d_model;
    L.F = p.d_ff;
    L.E = p.E;
    L.S = p.n_shared;
    L.k = p.k;
    L.C = (int)capacity_of(p);
    const long long slots = (long long)p.T * p.k;
    L.nchunks = (int)((slots + kScanChunk - 1) / kScanChunk);
    long long cap = slots + (long long)p.E * (kSegRows - 1);
    if (L.C >= 0) cap = std::min(cap, (long long)p.E * (((long long)L.C + kSegRows - 1) / kSegRows * kSegRows));
    L.rows_cap = (int)((cap + kSegRows - 1) / kSegRows * kSegRows);
    L.t_pad = (p.T + kSegRows - 1) / kSegRows * kSegRows;
    L.esz = (p.dtype == MOE_BF16) ? 2 : 4;
    L.tc_router = p.dtype == MOE_BF16 && !(p.flags & MOE_FLAG_FFMA_ROUTER);
    L.tc_rbwd = L.tc_router;
    L.r_bn = router_tc_bn(p.T, p.E);
    L.r_tiles = (p.E + L.r_bn - 1) / L.r_bn;
    L.e_pad = L.r_tiles * L.r_bn;
    L.r_ksplits = L.tc_router ? router_tc_ksplits(p.T, p.E, p.d_model) : 1;
    // one expert tile and no K split: the router GEMM's epilogue finishes the router;
    // otherwise (tensor-core logits) k_router_topk does, with its own column-sum rows
    L.r_fuse = L.tc_router && p.noisy_gating != 1 && L.r_tiles == 1 && L.r_ksplits == 1 && L.r_bn <= 32;
    L.n_rblk = (L.tc_router && !L.r_fuse) ? router_topk_blocks(p.T) : router_blocks(p.T);

    size_t o = kRegionAlign;  // header: [0] device error word, [1] scan arrival counter
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, kRegionAlign);
        return at;
    };
    const size_t split_bytes = 3 * sizeof(uint16_t) * (size_t)router_split_rows(L.E) * L.d;
    L.off_wsplit = take(L.tc_router ? split_bytes : 0);
    L.off_logits = take(sizeof(float) * (size_t)L.T * L.E * (L.r_ksplits > 1 ? L.r_ksplits + 1 : 1));
    const bool noisy = p.noisy_gating == 1;
    L.off_nsplit = take(noisy && L.tc_router ? split_bytes : 0);
    L.off_nlogits = take(noisy ? sizeof(float) * (size_t)L.T * L.E * L.r_ksplits : 0);
    // fused experts' scheduler words: tile counter, finished CTAs, one counter per routed
    // M-tile and, with shared experts, one per shared M-tile
    L.ffn_sync_n = 2 + L.rows_cap / kSegRows + (L.S > 0 ? L.t_pad / kSegRows : 0);
    L.off_ffn_sync = take(sizeof(unsigned) * L.ffn_sync_n);
    L.off_psum = take(sizeof(float) * L.n_rblk * L.E);
    L.off_psum_chunk = take(sizeof(float) * (size_t)L.nchunks * L.E);
    L.off_hist = take(sizeof(int32_t) * (size_t)L.nchunks * L.E);
    L.off_base = take(sizeof(int32_t) * (size_t)L.nchunks * L.E);
    L.off_rank = take(sizeof(int32_t) * (size_t)slots);
    L.off_slot_row = take(sizeof(int32_t) * (size_t)slots);
    L.off_kept = take(sizeof(int32_t) * L.E);
    L.off_row_off = take(sizeof(int32_t) * L.E);
    L.off_kept_off = take(sizeof(int32_t) * L.E);
    L.off_mtile = take(sizeof(int32_t) * (L.E + 1));
    L.off_xp = take(L.esz * (size_t)L.rows_cap * L.d);
    L.off_h = take(L.esz * (size_t)L.rows_cap * L.F);
    L.off_yp = take(L.esz * (size_t)L.rows_cap * L.d);
    L.off_row_token = take(sizeof(int32_t) * (size_t)L.rows_cap);
    L.off_row_gate = take(sizeof(float) * (size_t)L.rows_cap);
    L.off_hs = take(L.S > 0 ? L.esz * (size_t)L.t_pad * L.S * L.F : 0);
    L.off_ys = take(L.S > 0 ? L.esz * (size_t)L.t_pad * L.d : 0);
    const bool train = (p.flags & MOE_FLAG_TRAINING) != 0u;
    const bool swiglu = p.act == MOE_ACT_SWIGLU;
    auto bw = [&](size_t bytes) { return take(train ? bytes : 0); };
    L.off_bw_dgate = bw(sizeof(float) * (size_t)slots);
    L.off_bw_dl = bw(sizeof(float) * (size_t)L.T * L.E);
    L.off_bw_dn = bw(noisy ? sizeof(float) * (size_t)L.T * L.E : 0);
    L.off_bw_dxr = bw(sizeof(float) * (size_t)L.T * L.d);
    L.off_bw_dyp = bw(L.esz * (size_t)L.rows_cap * L.d);
    L.off_bw_z1 = bw(L.esz * (size_t)L.rows_cap * L.F);
    L.off_bw_z3 = bw(swiglu ? L.esz * (size_t)L.rows_cap * L.F : 0);
    L.off_bw_zs1 = bw(L.S > 0 ? L.esz * (size_t)L.T * L.S * L.F : 0);
    L.off_bw_zs3 = bw(L.S > 0 ? L.esz * (size_t)L.T * L.S * L.F : 0);
    L.off_bw_dxs = bw(L.S > 0 ? L.esz * (size_t)L.T * L.d : 0);
    L.e8 = (L.E + 7) / 8 * 8;
    L.r_nblk = noisy ? 8 : 4;
    const bool tcr = train && L.tc_rbwd;
    L.off_bw_dcat = take(tcr ? sizeof(uint16_t) * (size_t)L.T * L.r_nblk * L.e8 : 0);
    L.off_bw_wcat = take(tcr ? sizeof(uint16_t) * (size_t)L.r_nblk * L.e8 * L.d : 0);
    L.r_dw_splits = router_dw_splits(L.T, L.e8, L.d);
    L.off_bw_p = take(tcr ? sizeof(float) * 3 * (size_t)L.e8 * L.d * L.r_dw_splits * (noisy ? 2 : 1) : 0);
    L.total = o;
    return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t validate_io(const moe_params_t& p, const moe_inputs_t* in, const moe_outputs_t* out)
{
    if (in == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
    const bool swiglu = p.act == MOE_ACT_SWIGLU;
    // arrays with T rows may be NULL for an empty batch (an empty tensor has no storage)
    const bool rows = p.T > 0;
    if ((rows && !in->x) || !in->W_gate || !in->W1 || !in->W2) return MOE_ERR_INVALID_ARG;
    if (swiglu != (in->W3 != nullptr)) return MOE_ERR_INVALID_ARG;
    if (swiglu && (in->b1 || in->b2)) return MOE_ERR_INVALID_ARG;
    if ((rows && (!out->y || !out->expert_idx || !out->gates || !out->dropped)) || !out->counts || !out->aux)
        return MOE_ERR_INVALID_ARG;
    if (p.noisy_gating == 1 ? (!in->W_noise || (rows && !in->noise_eps))
                            : (in->W_noise || in->b_noise || in->noise_eps))
        return MOE_ERR_INVALID_ARG;
    if (p.weight_format != MOE_WEIGHTS_DTYPE ? (!in->W1_scale || !in->W2_scale || (swiglu != (in->W3_scale != nullptr)))
                                            : (in->W1_scale || in->W3_scale || in->W2_scale))
        return MOE_ERR_INVALID_ARG;
    const bool tc_router = p.dtype == MOE_BF16 && !(p.flags & MOE_FLAG_FFMA_ROUTER);
    if (in->router_weights && !tc_router) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {in->router_weights, in->x, in->W_gate, in->b_gate, in->W1, in->W3, in->W2, in->b1, in->b2,
                          out->y, out->expert_idx, out->gates, out->counts, out->dropped, out->aux,
                          out->logits, out->probs, out->perm_row, in->W_noise, in->b_noise, in->noise_eps,
                          in->W1_scale, in->W3_scale, in->W2_scale};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

struct DeviceCache {
    std::once_flag once;
    int sms = 0;
};
DeviceCache g_dev[64];

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    DeviceCache& c = g_dev[dev];
    std::call_once(c.once, [&] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) c.sms = n;
    });
    return c.sms;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// 2-D byte tensor map over a row-major [rows, cols] int8 matrix, box {64, box_rows},
// no swizzle (64-byte rows in shared memory), zero fill out of bounds.
// 2-D byte tensor map over a row-major [rows, cols] array, box {box_cols, box_rows},
// with the given swizzle (the box's rows are box_cols bytes), zero fill out of bounds.
bool encode_u8_2d_swizzled(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                           uint32_t box_rows, CUtensorMapSwizzle swz)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u8_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box {64, box_rows},
// 128-byte swizzle, zero fill out of bounds.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_bn(int N) { return N >= 256 ? 256 : 128; }

// PDL for every launch of a C-ABI call except its first one (whose predecessor in
// the stream may be the caller's own work).
bool take_pdl(Ctx& c)
{
    const bool p = c.pdl;
    c.pdl = true;
    return p;
}

moe_status_t prepare(const moe_params_t* params, const moe_inputs_t* in, moe_outputs_t* out, void* ws,
                     size_t ws_bytes, void* stream, Ctx& c, bool io_checked)
{
    moe_status_t s = validate_params(params);
    if (s != MOE_OK) return s;
    c.p = *params;
    s = io_checked ? MOE_OK : validate_io(c.p, in, out);
    if (s != MOE_OK) return s;
    c.in = in;
    c.out = out;
    c.L = make_layout(c.p);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < c.L.total) return MOE_ERR_WORKSPACE;
    c.ws = static_cast<char*>(ws);
    c.st = static_cast<cudaStream_t>(stream);
    c.sms = sm_count();
    if (c.sms <= 0) return MOE_ERR_CUDA;
    c.bf16 = c.p.dtype == MOE_BF16;
    if (c.L.T == 0) return MOE_OK;  // an empty batch: no kernel, no tensor map
    c.use_tc = c.bf16 && !(c.p.flags & MOE_FLAG_FFMA_EXPERTS);
    c.fused = c.use_tc && !(c.p.flags & MOE_FLAG_UNFUSED_EXPERTS);
    if (c.L.tc_router) {
        const Layout& L = c.L;
        // the split router weights: the caller's prepared buffer (gate, then noise) or the workspace
        const uint64_t srows = 3ull * router_split_rows(L.E);
        const size_t sbytes = 2 * srows * (size_t)L.d;
        const void* wsplit = in->router_weights ? in->router_weights : c.at<void>(L.off_wsplit);
        const void* nsplit = in->router_weights ? static_cast<const char*>(in->router_weights) + sbytes
                                                : c.at<void>(L.off_nsplit);
        if (!encode_bf16_2d(&c.mX, in->x, L.T, L.d, 128) || !encode_bf16_2d(&c.mW, wsplit, srows, L.d, 3 * L.r_bn))
            return MOE_ERR_UNSUPPORTED;
        if (c.p.noisy_gating == 1 && !encode_bf16_2d(&c.mWn, nsplit, srows, L.d, 3 * L.r_bn))
            return MOE_ERR_UNSUPPORTED;
    }
    // quantised expert weights: the transposed tensor-memory kernel (k_grouped_gemm_wq) for
    // layers whose experts hold at most 128 token rows each (the expert stage streams the
    // weights) and for every 4-bit layer; the 8-bit shared-memory converter kernel otherwise
    c.q8 = c.p.weight_format == MOE_WEIGHTS_INT8;
    c.wq = c.p.weight_format == MOE_WEIGHTS_INT4;
    if (c.q8 || c.wq) {
        const long long bound = c.L.C >= 0 ? std::min(c.L.C, c.L.T) : c.L.T;  // rows one expert can hold
        if (c.q8 && bound <= 128) c.wq = true;
    }
    if (c.wq) {
        const Layout& L = c.L;
        const bool gated = c.p.act == MOE_ACT_SWIGLU;
        // token rows per tile: enough for the rows an expert can hold (the capacity, or the
        // batch), but not far beyond what it holds on average, so that the token tile is not
        // mostly padding
        const long long avg = ((long long)L.T * L.k + L.E - 1) / L.E;
        const long long bound = L.C >= 0 ? std::min<long long>(L.C, L.T) : L.T;
        const long long est = std::min<long long>(bound, 2 * avg + 16);
        c.wq_bits = c.p.weight_format == MOE_WEIGHTS_INT4 ? 4 : 8;
        c.wq_nt = gemm_wq_tokens_tile((int)std::min<long long>(est, 1 << 30), gated);
        // one stage reads 128 bytes of each weight row (128 int8 or 256 int4 values)
        const uint32_t kb_bytes = 128;
        const CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B;
        const uint64_t dcols = (uint64_t)L.d * c.wq_bits / 8, fcols = (uint64_t)L.F * c.wq_bits / 8;
        bool ok = encode_u8_2d_swizzled(&c.mQ1, in->W1, (uint64_t)L.E * L.F, dcols, kb_bytes, 128, swz) &&
                  encode_u8_2d_swizzled(&c.mQ3, gated ? in->W3 : in->W1, (uint64_t)L.E * L.F, dcols, kb_bytes, 128,
                                        swz) &&
                  encode_u8_2d_swizzled(&c.mQ2, in->W2, (uint64_t)L.E * L.d, fcols, kb_bytes, 128, swz);
        if (L.rows_cap > 0)
            ok = ok && encode_bf16_2d(&c.mA1, c.at<void>(L.off_xp), L.rows_cap, L.d, c.wq_nt) &&
                 encode_bf16_2d(&c.mA2, c.at<void>(L.off_h), L.rows_cap, L.F, c.wq_nt);
        if (!ok) return MOE_ERR_UNSUPPORTED;
        c.q8 = false;
        c.use_tc = false;  // the quantised-weight kernels replace the bf16 tensor-core path
        c.fused = false;
    } else if (c.q8) {
        const Layout& L = c.L;
        const bool gated = c.p.act == MOE_ACT_SWIGLU;
        const uint32_t r1 = gated ? 128 : 256;
        bool ok = encode_u8_2d(&c.mQ1, in->W1, (uint64_t)L.E * L.F, L.d, r1) &&
                  encode_u8_2d(&c.mQ3, gated ? in->W3 : in->W1, (uint64_t)L.E * L.F, L.d, r1) &&
                  encode_u8_2d(&c.mQ2, in->W2, (uint64_t)L.E * L.d, L.F, 256);
        if (L.rows_cap > 0)
            ok = ok && encode_bf16_2d(&c.mA1, c.at<void>(L.off_xp), L.rows_cap, L.d, 128) &&
                 encode_bf16_2d(&c.mA2, c.at<void>(L.off_h), L.rows_cap, L.F, 128);
        if (!ok) return MOE_ERR_UNSUPPORTED;
        c.use_tc = false;  // the int8 kernels replace the bf16 tensor-core path
        c.fused = false;
    } else if (c.use_tc) {
        const Layout& L = c.L;
        const bool gated = c.p.act == MOE_ACT_SWIGLU;
        // a top-1 layer without shared experts or the residual on every token: each kept
        // row is one token's whole routed output, so the fused kernel's GEMM2 epilogue
        // scales it by the gate and writes y (the arithmetic k_combine would apply), and
        // the dispatch copies the dropped tokens' x; training keeps Yp for the backward
        c.direct_y = c.fused && c.p.k == 1 && L.S == 0 && c.p.residual_mode == 0 &&
                     !(c.p.flags & MOE_FLAG_TRAINING);
        c.bn1 = c.fused || gated ? 256 : pick_bn(L.F);
        c.bn2 = c.fused ? 256 : pick_bn(L.d);
        const int b1_rows = gated ? c.bn1 / 2 : c.bn1;
        const uint64_t ES = (uint64_t)(L.E + L.S);
        bool ok = encode_bf16_2d(&c.mB1, in->W1, ES * L.F, L.d, b1_rows) &&
                  encode_bf16_2d(&c.mB2, in->W2, ES * L.d, L.F, c.bn2);
        ok = ok && encode_bf16_2d(&c.mB3, gated ? in->W3 : in->W1, ES * L.F, L.d, b1_rows);
        if (L.rows_cap > 0)
            ok = ok && encode_bf16_2d(&c.mA1, c.at<void>(L.off_xp), L.rows_cap, L.d, 128) &&
                 encode_bf16_2d(&c.mA2, c.at<void>(L.off_h), L.rows_cap, L.F, 128) &&
                 encode_bf16_2d(&c.mA1p, c.at<void>(L.off_xp), L.rows_cap, L.d, kABoxRows) &&
                 encode_bf16_2d(&c.mA2p, c.at<void>(L.off_h), L.rows_cap, L.F, kABoxRows);
        if (L.S > 0)
            ok = ok && encode_bf16_2d(&c.mAs1, in->x, L.T, L.d, 128) &&
                 encode_bf16_2d(&c.mAs2, c.at<void>(L.off_hs), L.t_pad, (uint64_t)L.S * L.F, 128) &&
                 encode_bf16_2d(&c.mAs1p, in->x, L.T, L.d, kABoxRows) &&
                 encode_bf16_2d(&c.mAs2p, c.at<void>(L.off_hs), L.t_pad, (uint64_t)L.S * L.F, kABoxRows);
        if (!ok) return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t stage_router(Ctx& c)
{
    if (c.L.T == 0) return MOE_OK;
    RouterArgs a{};
    a.x = c.in->x;
    a.Wg = c.in->W_gate;
    a.bg = c.in->b_gate;
    a.T = c.L.T;
    a.d = c.L.d;
    a.E = c.L.E;
    a.k = c.L.k;
    a.renormalize = c.p.renormalize;
    a.idx = c.out->expert_idx;
    a.gates = c.out->gates;
    a.logits = c.out->logits;
    a.probs = c.out->probs;
    a.psum_part = c.at<float>(c.L.off_psum);
    a.scan_done = c.scan_done();
    const bool noisy = c.p.noisy_gating == 1;
    if (noisy) {
        a.noise_parts = c.at<float>(c.L.off_nlogits);
        a.bn = c.in->b_noise;
        a.eps = c.in->noise_eps;
        a.min_std = c.p.noise_min_std;
    }
    if (!c.L.tc_router) {
        // training keeps the logits for the backward pass
        if (a.logits == nullptr && (c.p.flags & MOE_FLAG_TRAINING)) a.logits = c.at<float>(c.L.off_logits);
        cudaError_t e = cudaSuccess;
        if (noisy) {  // noise projection x W_noise^T first, then the routing pass adds the noise
            RouterArgs r = a;
            r.Wg = c.in->W_noise;
            r.bg = nullptr;
            r.raw_out = c.at<float>(c.L.off_nlogits);
            e = launch_router(r, c.bf16, c.st, take_pdl(c));
        }
        if (e == cudaSuccess) e = launch_router(a, c.bf16, c.st, take_pdl(c));
        return cuda_status(e);
    }
    // tensor-core logits into the caller's logits buffer (or the workspace), then top-k;
    // with split K, partial sums go to the workspace and the top-k kernel adds them
    if (a.logits == nullptr) a.logits = c.at<float>(c.L.off_logits);
    const bool split = c.L.r_ksplits > 1;
    float* parts = c.at<float>(c.L.off_logits) + (size_t)c.L.T * c.L.E;
    a.logit_parts = split ? parts : nullptr;
    a.k_splits = c.L.r_ksplits;
    RouterGemmArgs g{};
    g.T = c.L.T;
    g.d = c.L.d;
    g.E = c.L.E;
    g.E_pad = c.L.e_pad;
    g.n_tiles = c.L.r_tiles;
    g.k_splits = c.L.r_ksplits;
    g.bg = c.in->b_gate;
    g.logits = split ? parts : a.logits;
    g.err = c.err();
    g.fuse = c.L.r_fuse ? 1 : 0;
    if (g.fuse) {
        g.k = a.k;
        g.renormalize = a.renormalize;
        g.idx = a.idx;
        g.gates = a.gates;
        g.probs = a.probs;
        g.psum_part = a.psum_part;
        g.scan_done = a.scan_done;
    }
    const bool prepared = c.in->router_weights != nullptr;  // split once by the caller
    cudaError_t e = prepared ? cudaSuccess
                             : launch_split_wgate(c.in->W_gate, c.L.E, c.L.d, c.at<void>(c.L.off_wsplit), c.sms, c.st,
                                                  take_pdl(c));
    if (e == cudaSuccess) e = launch_router_logits_tc(c.mX, c.mW, g, c.L.r_bn, c.sms, c.st, take_pdl(c));
    if (noisy) {  // the same GEMM on W_noise, without bias, into the noise-logit partials
        RouterGemmArgs gn = g;
        gn.bg = nullptr;
        gn.logits = c.at<float>(c.L.off_nlogits);
        if (e == cudaSuccess)
            e = prepared ? cudaSuccess
                         : launch_split_wgate(c.in->W_noise, c.L.E, c.L.d, c.at<void>(c.L.off_nsplit), c.sms, c.st,
                                              take_pdl(c));
        if (e == cudaSuccess) e = launch_router_logits_tc(c.mX, c.mWn, gn, c.L.r_bn, c.sms, c.st, take_pdl(c));
    }
    if (e == cudaSuccess && !g.fuse) e = launch_router_topk(a, c.st);
    return cuda_status(e);
}

moe_status_t stage_dispatch(Ctx& c)
{
    if (c.L.T == 0) {  // an empty batch: no expert receives a token, the statistic is 0
        cudaError_t e = cudaMemsetAsync(c.out->counts, 0, sizeof(int32_t) * c.L.E, c.st);
        if (e == cudaSuccess) e = cudaMemsetAsync(c.out->aux, 0, sizeof(float), c.st);
        return cuda_status(e);
    }
    DispatchArgs a{};
    a.idx = c.out->expert_idx;
    a.gates = c.out->gates;
    a.T = c.L.T;
    a.k = c.L.k;
    a.E = c.L.E;
    a.C = c.L.C;
    a.nchunks = c.L.nchunks;
    a.n_router_blocks = c.L.n_rblk;
    a.psum_part = c.at<float>(c.L.off_psum);
    a.psum_chunk = c.at<float>(c.L.off_psum_chunk);
    a.local_rank = c.at<int32_t>(c.L.off_rank);
    a.chunk_hist = c.at<int32_t>(c.L.off_hist);
    a.chunk_base = c.at<int32_t>(c.L.off_base);
    a.scan_done = c.scan_done();
    a.counts = c.out->counts;
    a.kept = c.at<int32_t>(c.L.off_kept);
    a.row_off = c.at<int32_t>(c.L.off_row_off);
    a.kept_off = c.at<int32_t>(c.L.off_kept_off);
    a.mtile_off = c.at<int32_t>(c.L.off_mtile);
    a.aux = c.out->aux;
    a.x = c.in->x;
    a.xp = c.at<void>(c.L.off_xp);
    a.row_bytes = (int)(c.L.d * c.L.esz);
    a.dropped = c.out->dropped;
    a.perm_row = c.out->perm_row;
    a.slot_row = c.at<int32_t>(c.L.off_slot_row);
    a.ffn_sync = c.at<unsigned>(c.L.off_ffn_sync);
    a.ffn_sync_n = c.L.ffn_sync_n;
    if (c.direct_y) {
        a.row_token = c.at<int32_t>(c.L.off_row_token);
        a.row_gate = c.at<float>(c.L.off_row_gate);
        a.y_pass = c.out->y;
    }
    return cuda_status(launch_dispatch(a, c.sms, c.st, take_pdl(c)));
}

moe_status_t stage_gemm(Ctx& c)
{
    if (c.L.T == 0) return MOE_OK;
    const Layout& L = c.L;
    const bool gated = c.p.act == MOE_ACT_SWIGLU;
    const int act1 = c.p.act;  // moe_act_t values equal the kernels' ActKind values
    GroupedGemmArgs g1{};
    g1.mtile_off = c.at<int>(L.off_mtile);
    g1.row_off = c.at<int>(L.off_row_off);
    g1.rows = c.at<int>(L.off_kept);
    g1.G = L.E;
    g1.N = L.F;
    g1.K = L.d;
    g1.k_segments = 1;
    g1.b_rows_per_group = L.F;
    g1.b_group0 = 0;
    g1.out = c.at<void>(L.off_h);
    g1.ldo = L.F;
    g1.bias = c.in->b1;
    g1.a_rows_alloc = L.rows_cap;
    g1.err = c.err();

    GroupedGemmArgs g2 = g1;
    g2.N = L.d;
    g2.K = L.F;
    g2.b_rows_per_group = L.d;
    g2.out = c.at<void>(L.off_yp);
    g2.ldo = L.d;
    g2.bias = c.in->b2;

    // shared experts: one group of all T tokens, hidden S*F (concatenated experts)
    GroupedGemmArgs s1 = g1;
    s1.mtile_off = nullptr;
    s1.row_off = nullptr;
    s1.rows = nullptr;
    s1.G = 1;
    s1.fixed_rows = L.T;
    s1.N = L.S * L.F;
    s1.b_group0 = L.E;
    s1.out = c.at<void>(L.off_hs);
    s1.ldo = L.S * L.F;
    s1.a_rows_alloc = L.T;
    GroupedGemmArgs s2 = g2;
    s2.mtile_off = nullptr;
    s2.row_off = nullptr;
    s2.rows = nullptr;
    s2.G = 1;
    s2.fixed_rows = L.T;
    s2.k_segments = L.S;
    s2.b_group0 = L.E;
    s2.out = c.at<void>(L.off_ys);
    s2.a_rows_alloc = L.T;

    const int mt_routed = c.routed_experts ? L.rows_cap / kSegRows : 0;
    const int mt_shared = L.t_pad / kSegRows;
    auto grid_for = [&](int tiles, int per_sm) { return std::max(1, std::min(tiles, c.sms * per_sm)); };
    cudaError_t e = cudaSuccess;
    // training: the first layer also keeps its pre-activations for the backward pass
    // (relu's derivative comes from H itself)
    const bool save = (c.p.flags & MOE_FLAG_TRAINING) && c.p.act != MOE_ACT_RELU;
    if (c.wq) {
        if (mt_routed == 0) return MOE_OK;
        GroupedGemmWqArgs w1{};
        w1.row_off = g1.row_off;
        w1.rows = g1.rows;
        w1.G = L.E;
        w1.N = L.F;
        w1.n_tiles = gemm_wq_weight_tiles(L.F, act1, c.wq_nt);
        w1.K = L.d;
        w1.b_rows_per_group = L.F;
        w1.out = g1.out;
        w1.ldo = L.F;
        w1.bias = c.in->b1;
        w1.scale = c.in->W1_scale;
        w1.scale3 = c.in->W3_scale;
        w1.err = c.err();
        GroupedGemmWqArgs w2 = w1;
        w2.N = L.d;
        w2.n_tiles = gemm_wq_weight_tiles(L.d, kActNone, c.wq_nt);
        w2.K = L.F;
        w2.b_rows_per_group = L.d;
        w2.out = g2.out;
        w2.ldo = L.d;
        w2.bias = c.in->b2;
        w2.scale = c.in->W2_scale;
        w2.scale3 = nullptr;
        const int token_tiles = L.rows_cap / c.wq_nt;  // bound: segments are padded to 128 rows
        e = launch_gemm_wq(c.mA1, c.mQ1, c.mQ3, w1, c.wq_bits, act1, c.wq_nt,
                           grid_for(token_tiles * w1.n_tiles, 1), c.st, take_pdl(c));
        if (e == cudaSuccess)
            e = launch_gemm_wq(c.mA2, c.mQ2, c.mQ2, w2, c.wq_bits, kActNone, c.wq_nt,
                               grid_for(token_tiles * w2.n_tiles, 1), c.st, take_pdl(c));
        return cuda_status(e);
    }
    if (c.q8) {
        if (mt_routed == 0) return MOE_OK;
        GroupedGemmQ8Args q1{};
        q1.mtile_off = g1.mtile_off;
        q1.row_off = g1.row_off;
        q1.rows = g1.rows;
        q1.G = L.E;
        q1.N = L.F;
        q1.n_tiles = ceil_div(L.F, gated ? 128 : 256);
        q1.K = L.d;
        q1.b_rows_per_group = L.F;
        q1.out = g1.out;
        q1.ldo = L.F;
        q1.bias = c.in->b1;
        q1.scale = c.in->W1_scale;
        q1.scale3 = c.in->W3_scale;
        q1.err = c.err();
        GroupedGemmQ8Args q2 = q1;
        q2.N = L.d;
        q2.n_tiles = ceil_div(L.d, 256);
        q2.K = L.F;
        q2.b_rows_per_group = L.d;
        q2.out = g2.out;
        q2.ldo = L.d;
        q2.bias = c.in->b2;
        q2.scale = c.in->W2_scale;
        q2.scale3 = nullptr;
        e = launch_gemm_q8(c.mA1, c.mQ1, c.mQ3, q1, act1, grid_for(mt_routed * q1.n_tiles, 1), c.st, take_pdl(c));
        if (e == cudaSuccess)
            e = launch_gemm_q8(c.mA2, c.mQ2, c.mQ2, q2, kActNone, grid_for(mt_routed * q2.n_tiles, 1), c.st,
                               take_pdl(c));
        return cuda_status(e);
    }
    if (save && c.use_tc) {
        g1.z1 = c.at<void>(L.off_bw_z1);
        g1.z3 = gated ? c.at<void>(L.off_bw_z3) : nullptr;
        if (L.S > 0) {
            s1.z1 = c.at<void>(L.off_bw_zs1);
            s1.z3 = c.at<void>(L.off_bw_zs3);
        }
    }
    if (c.use_tc) {
        const int out1 = gated ? c.bn1 / 2 : c.bn1;
        g1.n_tiles = ceil_div(L.F, out1);
        g2.n_tiles = ceil_div(L.d, c.bn2);
        // the shared experts join the fused kernel's tile list when their GEMM2 K blocks
        // never straddle two experts (d_ff a multiple of 64)
        const bool fold_shared = c.fused && L.S > 0 && mt_routed > 0 && gated && L.F % 64 == 0;
        if (mt_routed > 0 && c.fused) {
            FusedFfnArgs f{};
            f.mtile_off = g1.mtile_off;
            f.row_off = g1.row_off;
            f.rows = g1.rows;
            f.G = L.E;
            f.N1 = L.F;
            f.n_tiles1 = g1.n_tiles;
            f.K1 = L.d;
            f.N2 = L.d;
            f.n_tiles2 = g2.n_tiles;
            f.K2 = L.F;
            f.b1_rows_per_group = L.F;
            f.b2_rows_per_group = L.d;
            f.h = g1.out;
            f.ldh = L.F;
            f.yp = g2.out;
            f.ldy = L.d;
            f.bias1 = c.in->b1;
            f.bias2 = c.in->b2;
            f.z1 = g1.z1;
            f.z3 = g1.z3;
            unsigned* sync = c.at<unsigned>(L.off_ffn_sync);
            f.tile_ctr = sync;
            f.ctas_done = sync + 1;
            f.mt_done = sync + 2;
            f.mt_max = L.ffn_sync_n - 2;
            f.err = c.err();
            if (c.direct_y) {
                f.y = c.out->y;
                f.row_token = c.at<int32_t>(L.off_row_token);
                f.row_gate = c.at<float>(L.off_row_gate);
            }
            int tiles = mt_routed * (g1.n_tiles + g2.n_tiles);
            if (fold_shared) {
                f.S = L.S;
                f.shared_rows = L.T;
                f.mt_s = mt_shared;
                f.n_tiles_s1 = ceil_div(L.S * L.F, out1);
                f.b1_row0 = L.E * L.F;
                f.b2_group0 = L.E;
                f.seg_k2 = L.F;
                f.hs = s1.out;
                f.ldhs = L.S * L.F;
                f.ys = s2.out;
                f.zs1 = s1.z1;
                f.zs3 = s1.z3;
                f.mt_s0 = L.rows_cap / kSegRows;
                tiles += mt_shared * (f.n_tiles_s1 + g2.n_tiles);
            }
            // experts of about one M-tile (the layer streams its weights): most M-tiles are
            // partial, so load only their valid rows
            f.partial_a = mt_routed <= L.E ? 1 : 0;
            const CUtensorMap maps[11] = {c.mA1,  c.mB1,  c.mB3,  c.mA2,  c.mB2, c.mAs1,
                                          c.mAs2, c.mA1p, c.mA2p, c.mAs1p, c.mAs2p};
            e = launch_ffn_fused_tc(maps, f, act1, grid_for(tiles, 1), c.st, take_pdl(c));
        } else if (mt_routed > 0) {
            e = launch_gemm_tc(c.mA1, c.mB1, c.mB3, g1, act1, c.bn1, grid_for(mt_routed * g1.n_tiles, 1), c.st,
                               take_pdl(c));
            if (e == cudaSuccess)
                e = launch_gemm_tc(c.mA2, c.mB2, c.mB2, g2, kActNone, c.bn2, grid_for(mt_routed * g2.n_tiles, 1),
                                   c.st, take_pdl(c));
        }
        if (e == cudaSuccess && L.S > 0 && !fold_shared) {
            s1.n_tiles = ceil_div(s1.N, out1);
            s2.n_tiles = ceil_div(L.d, c.bn2);
            e = launch_gemm_tc(c.mAs1, c.mB1, c.mB3, s1, act1, c.bn1, grid_for(mt_shared * s1.n_tiles, 1), c.st,
                               take_pdl(c));
            if (e == cudaSuccess)
                e = launch_gemm_tc(c.mAs2, c.mB2, c.mB2, s2, kActNone, c.bn2, grid_for(mt_shared * s2.n_tiles, 1),
                                   c.st, take_pdl(c));
        }
    } else {
        g1.n_tiles = ceil_div(L.F, kFfmaTileN);
        g2.n_tiles = ceil_div(L.d, kFfmaTileN);
        if (mt_routed > 0) {
            e = launch_gemm_ffma(c.at<void>(L.off_xp), L.d, c.in->W1, c.in->W3, L.d, g1, act1, c.bf16,
                                 grid_for(mt_routed * g1.n_tiles, 4), c.st, take_pdl(c));
            if (e == cudaSuccess)
                e = launch_gemm_ffma(c.at<void>(L.off_h), L.F, c.in->W2, nullptr, L.F, g2, kActNone, c.bf16,
                                     grid_for(mt_routed * g2.n_tiles, 4), c.st, take_pdl(c));
        }
        if (e == cudaSuccess && L.S > 0) {
            s1.n_tiles = ceil_div(s1.N, kFfmaTileN);
            s2.n_tiles = ceil_div(L.d, kFfmaTileN);
            e = launch_gemm_ffma(c.in->x, L.d, c.in->W1, c.in->W3, L.d, s1, act1, c.bf16,
                                 grid_for(mt_shared * s1.n_tiles, 4), c.st, take_pdl(c));
            if (e == cudaSuccess)
                e = launch_gemm_ffma(c.at<void>(L.off_hs), L.S * L.F, c.in->W2, nullptr, L.F, s2, kActNone,
                                     c.bf16, grid_for(mt_shared * s2.n_tiles, 4), c.st, take_pdl(c));
        }
    }
    return cuda_status(e);
}

moe_status_t stage_combine(Ctx& c)
{
    if (c.L.T == 0) return MOE_OK;
    if (c.direct_y) return MOE_OK;  // the expert stage and the dispatch wrote y
    CombineArgs a{};
    a.yp = c.at<void>(c.L.off_yp);
    a.ys = c.L.S > 0 ? c.at<void>(c.L.off_ys) : nullptr;
    a.x = c.in->x;
    a.slot_row = c.at<int32_t>(c.L.off_slot_row);
    a.gates = c.out->gates;
    a.y = c.out->y;
    a.T = c.L.T;
    a.k = c.L.k;
    a.d = c.L.d;
    a.residual_mode = c.p.residual_mode;
    return cuda_status(launch_combine(a, c.bf16, c.sms, c.st, take_pdl(c)));
}

using StageFn = moe_status_t (*)(Ctx&);

moe_status_t run_stages(const moe_params_t* params, const moe_inputs_t* in, moe_outputs_t* out, void* ws,
                        size_t ws_bytes, void* stream, std::initializer_list<StageFn> stages)
{
    Ctx c;
    moe_status_t s = prepare(params, in, out, ws, ws_bytes, stream, c);
    if (s != MOE_OK) return s;
    for (StageFn f : stages) {
        s = f(c);
        if (s != MOE_OK) return s;
    }
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// Backward pass

moe_status_t validate_grads(const moe_params_t& p, const moe_inputs_t* in, const void* dy, float d_aux,
                            const moe_grads_t* g)
{
    const bool rows = p.T > 0;  // dy and dx may be NULL for an empty batch
    if (g == nullptr || (rows && dy == nullptr) || !aligned16(dy) || !std::isfinite(d_aux)) return MOE_ERR_INVALID_ARG;
    if ((rows && !g->dx) || !g->dW_gate || !g->dW1 || !g->dW2) return MOE_ERR_INVALID_ARG;
    const bool swiglu = p.act == MOE_ACT_SWIGLU, noisy = p.noisy_gating == 1;
    if ((g->dW3 != nullptr) != swiglu || (g->db_gate != nullptr) != (in->b_gate != nullptr) ||
        (g->db1 != nullptr) != (in->b1 != nullptr) || (g->db2 != nullptr) != (in->b2 != nullptr) ||
        (g->dW_noise != nullptr) != noisy || (g->db_noise != nullptr) != (noisy && in->b_noise != nullptr))
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {g->dx, g->dW_gate, g->db_gate, g->dW1, g->dW3, g->dW2, g->db1, g->db2, g->dW_noise,
                          g->db_noise};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

const void* offset_elems(const void* p, size_t n, size_t esz)
{
    return p == nullptr ? nullptr : static_cast<const char*>(p) + n * esz;
}

// Router weight and input gradients on the tensor core (bf16 layers): split the
// fp32 logit gradients into exact bf16 terms, then one row-mode GEMM for the input
// gradient and one token-reduction GEMM (fp32 partials, summed) per weight.
cudaError_t router_bwd_tc(Ctx& c, const float* dl, const float* dn, float* dxr, const moe_grads_t* gr)
{
    const Layout& L = c.L;
    const bool noisy = dn != nullptr;
    void* dcat = c.at<void>(L.off_bw_dcat);
    void* wcat = c.at<void>(L.off_bw_wcat);
    float* P = c.at<float>(L.off_bw_p);
    const int W = L.r_nblk * L.e8;
    cudaError_t e = launch_split_grad(dl, dn, L.T, L.E, L.e8, L.r_nblk, dcat, c.sms, c.st, take_pdl(c));
    if (e == cudaSuccess)
        e = launch_split_wcat(c.in->W_gate, noisy ? c.in->W_noise : nullptr, L.E, L.e8, L.d, L.r_nblk, wcat, c.sms,
                              c.st, take_pdl(c));
    CUtensorMap kD, mD, mW, mX;
    if (!encode_bf16_2d(&kD, dcat, L.T, W, 128) || !encode_bf16_2d(&mD, dcat, L.T, W, 64) ||
        !encode_bf16_2d(&mW, wcat, W, L.d, 64) || !encode_bf16_2d(&mX, c.in->x, L.T, L.d, 64))
        return cudaErrorInvalidValue;
    auto grid_for = [&](long long tiles) { return (int)std::max(1ll, std::min(tiles, (long long)c.sms)); };
    {
        BwdTcArgs a{};  // dx_router = D Wcat
        a.G = 1;
        a.fixed_rows = L.T;
        a.N = L.d;
        a.K = W;
        a.C = dxr;
        a.ldc = L.d;
        a.err = c.err();
        const CUtensorMap maps[4] = {kD, mW, kD, mW};
        if (e == cudaSuccess)
            e = launch_gemm_bwd_tc(maps, a, kBwdRows, kEpiStoreF32,
                                   grid_for((long long)ceil_div(L.T, 128) * ceil_div(L.d, 256)), c.st, take_pdl(c));
    }
    for (int which = 0; which < (noisy ? 2 : 1); ++which) {
        // partials [3 E8, d] of dW = dl^T x (dn^T x), one per split term and per token split
        const int splits = L.r_dw_splits;
        BwdTcArgs a{};
        a.G = 1;
        a.fixed_rows = L.T;
        // split boundaries on 64-row K blocks, so no block reads into the next split
        a.split_rows = splits > 1 ? ceil_div(ceil_div(L.T, splits), 64) * 64 : 0;
        a.M = 3 * L.e8;
        a.N = L.d;
        a.a_col0 = which * 4 * L.e8;
        float* Pw = P + (size_t)which * 3 * L.e8 * L.d * splits;
        a.C = Pw;
        a.c_gs = 3ll * L.e8 * L.d;
        a.ldc = L.d;
        a.err = c.err();
        const int n_split = splits > 1 ? ceil_div(L.T, a.split_rows) : 1;
        const CUtensorMap maps[4] = {mD, mX, mD, mX};
        if (e == cudaSuccess)
            e = launch_gemm_bwd_tc(maps, a, kBwdReduce, kEpiStoreF32,
                                   grid_for((long long)n_split * ceil_div(a.M, 128) * ceil_div(L.d, 256)), c.st,
                                   take_pdl(c));
        if (e == cudaSuccess)
            e = launch_sum3(Pw, n_split, L.E, L.e8, L.d, which ? gr->dW_noise : gr->dW_gate, c.sms, c.st,
                            take_pdl(c));
    }
    return e;
}

// Routed and shared experts' backward on the tensor core (bf16 layers).
cudaError_t experts_bwd_tc(Ctx& c, const void* dy, const moe_grads_t* gr)
{
    const Layout& L = c.L;
    const size_t esz = L.esz;
    const bool swiglu = c.p.act == MOE_ACT_SWIGLU;
    void* dyp = c.at<void>(L.off_bw_dyp);
    void* z1 = c.at<void>(L.off_bw_z1);
    void* z3 = swiglu ? c.at<void>(L.off_bw_z3) : nullptr;
    void* h = c.at<void>(L.off_h);
    void* xp = c.at<void>(L.off_xp);
    const int* mtile = c.at<int>(L.off_mtile);
    const int* row_off = c.at<int>(L.off_row_off);
    const int* kept = c.at<int>(L.off_kept);
    const uint64_t R = (uint64_t)L.rows_cap, ES = (uint64_t)(L.E + L.S), SF = (uint64_t)L.S * L.F;
    const int mt_routed = L.rows_cap / kSegRows;
    auto grid_for = [&](long long tiles) { return (int)std::max(1ll, std::min(tiles, (long long)c.sms)); };
    auto tiles = [](int M, int N) { return (long long)ceil_div(M, 128) * ceil_div(N, 256); };

    // tensor maps: K-major A (box 64 x 128) and MN-major operands (box 64 x 64)
    CUtensorMap kDyp, kZ1, kZ3, mDyp, mZ1, mZ3, mH, mXp, mW2, mW1, mW3;
    bool ok = true;
    if (R > 0)
        ok = encode_bf16_2d(&kDyp, dyp, R, L.d, 128) && encode_bf16_2d(&kZ1, z1, R, L.F, 128) &&
             encode_bf16_2d(&mDyp, dyp, R, L.d, 64) && encode_bf16_2d(&mZ1, z1, R, L.F, 64) &&
             encode_bf16_2d(&mH, h, R, L.F, 64) && encode_bf16_2d(&mXp, xp, R, L.d, 64) &&
             (!swiglu || (encode_bf16_2d(&kZ3, z3, R, L.F, 128) && encode_bf16_2d(&mZ3, z3, R, L.F, 64)));
    ok = ok && encode_bf16_2d(&mW2, c.in->W2, ES * L.d, L.F, 64) && encode_bf16_2d(&mW1, c.in->W1, ES * L.F, L.d, 64) &&
         (!swiglu || encode_bf16_2d(&mW3, c.in->W3, ES * L.F, L.d, 64));
    if (!ok) return cudaErrorInvalidValue;
    if (!swiglu) {
        kZ3 = kZ1;
        mZ3 = mZ1;
        mW3 = mW1;
    }

    cudaError_t e = cudaSuccess;
    auto bwd = [&](const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a2, const CUtensorMap& b2,
                   const BwdTcArgs& args, int mode, int epi, long long n_tiles) {
        const CUtensorMap maps[4] = {a, b, a2, b2};
        if (e == cudaSuccess) e = launch_gemm_bwd_tc(maps, args, mode, epi, grid_for(n_tiles), c.st, take_pdl(c));
    };
    BwdTcArgs rows{};  // row-grouped (dgrad) products over the expert segments
    rows.mtile_off = mtile;
    rows.row_off = row_off;
    rows.rows = kept;
    rows.G = L.E;
    rows.err = c.err();
    BwdTcArgs red = rows;  // products reduced over each segment's rows (wgrad)
    red.mtile_off = nullptr;

    if (R > 0) {
        // the 64-row K blocks of the reductions read up to 63 rows past each segment's
        // kept rows: make them zero in every operand
        ZeroPadArgs zp{};
        zp.row_off = row_off;
        zp.rows = kept;
        zp.G = L.E;
        zp.buf[0] = dyp;
        zp.buf[1] = h;
        zp.buf[2] = xp;
        zp.row_bytes[0] = (int)(L.d * esz);
        zp.row_bytes[1] = (int)(L.F * esz);
        zp.row_bytes[2] = (int)(L.d * esz);
        e = launch_zero_pad_rows(zp, c.sms, c.st, take_pdl(c));
    }
    {
        BwdTcArgs a = red;  // dW2_e = dYp_e^T H_e
        a.M = L.d;
        a.N = L.F;
        a.C = gr->dW2;
        a.ldc = L.F;
        a.c_gs = (long long)L.d * L.F;
        if (R > 0) bwd(mDyp, mH, mDyp, mH, a, kBwdReduce, kEpiStore, L.E * tiles(a.M, a.N));
        else if (e == cudaSuccess) e = cudaMemsetAsync(gr->dW2, 0, esz * L.E * L.d * L.F, c.st);
    }
    if (gr->db2 && e == cudaSuccess) {
        ColsumArgs s{};
        s.A = dyp;
        s.lda = L.d;
        s.row_off = row_off;
        s.rows = kept;
        s.G = L.E;
        s.N = L.d;
        s.out = gr->db2;
        e = launch_colsum(s, kBwdTypesBf16, c.sms, c.st, take_pdl(c));
    }
    if (mt_routed > 0) {
        BwdTcArgs a = rows;  // dH = dYp W2_e with the activation backward
        a.N = L.F;
        a.K = L.d;
        a.b_rows_per_group = L.d;
        a.C = z1;
        a.ldc = L.F;
        int epi;
        if (c.p.act == MOE_ACT_RELU) {
            epi = kEpiReluBwd;
            a.e1 = h;
        } else if (swiglu) {
            epi = kEpiSwigluBwd;
            a.e1 = z1;
            a.e2 = z3;
            a.C2 = z3;
        } else {
            epi = c.p.act == MOE_ACT_GELU_TANH ? kEpiGeluTanhBwd : kEpiGeluErfBwd;
            a.e1 = z1;
        }
        bwd(kDyp, mW2, kDyp, mW2, a, kBwdRows, epi, (long long)mt_routed * ceil_div(a.N, 256));
    }
    {
        BwdTcArgs a = red;  // dW1_e = dZ1_e^T Xp_e, dW3_e = dZ3_e^T Xp_e
        a.M = L.F;
        a.N = L.d;
        a.C = gr->dW1;
        a.ldc = L.d;
        a.c_gs = (long long)L.F * L.d;
        if (R > 0) {
            bwd(mZ1, mXp, mZ1, mXp, a, kBwdReduce, kEpiStore, L.E * tiles(a.M, a.N));
            if (swiglu) {
                a.C = gr->dW3;
                bwd(mZ3, mXp, mZ3, mXp, a, kBwdReduce, kEpiStore, L.E * tiles(a.M, a.N));
            }
        } else {
            if (e == cudaSuccess) e = cudaMemsetAsync(gr->dW1, 0, esz * L.E * L.F * L.d, c.st);
            if (swiglu && e == cudaSuccess) e = cudaMemsetAsync(gr->dW3, 0, esz * L.E * L.F * L.d, c.st);
        }
    }
    if (gr->db1 && e == cudaSuccess) {
        ColsumArgs s{};
        s.A = z1;
        s.lda = L.F;
        s.row_off = row_off;
        s.rows = kept;
        s.G = L.E;
        s.N = L.F;
        s.out = gr->db1;
        e = launch_colsum(s, kBwdTypesBf16, c.sms, c.st, take_pdl(c));
    }
    if (mt_routed > 0) {
        BwdTcArgs a = rows;  // dXp = dZ1 W1_e (+ dZ3 W3_e), into the dYp buffer
        a.N = L.d;
        a.K = L.F;
        a.b_rows_per_group = L.F;
        a.two_seg = swiglu ? 1 : 0;
        a.C = dyp;
        a.ldc = L.d;
        bwd(kZ1, mW1, kZ3, mW3, a, kBwdRows, kEpiStore, (long long)mt_routed * ceil_div(a.N, 256));
    }

    if (L.S > 0) {
        // shared experts: one group of all T tokens, gate 1, SwiGLU, hidden S*F
        void* zs1 = c.at<void>(L.off_bw_zs1);
        void* zs3 = c.at<void>(L.off_bw_zs3);
        void* dxs = c.at<void>(L.off_bw_dxs);
        const uint64_t T = (uint64_t)L.T;
        CUtensorMap kDy, mDy, kZs1, kZs3, mZs1, mZs3, mHs, mX;
        ok = encode_bf16_2d(&kDy, dy, T, L.d, 128) && encode_bf16_2d(&mDy, dy, T, L.d, 64) &&
             encode_bf16_2d(&kZs1, zs1, T, SF, 128) && encode_bf16_2d(&kZs3, zs3, T, SF, 128) &&
             encode_bf16_2d(&mZs1, zs1, T, SF, 64) && encode_bf16_2d(&mZs3, zs3, T, SF, 64) &&
             encode_bf16_2d(&mHs, c.at<void>(L.off_hs), T, SF, 64) && encode_bf16_2d(&mX, c.in->x, T, L.d, 64);
        if (!ok) return cudaErrorInvalidValue;
        BwdTcArgs f{};
        f.G = 1;
        f.fixed_rows = L.T;
        f.err = c.err();
        for (int sh = 0; sh < L.S; ++sh) {
            BwdTcArgs w = f;  // dW2_s = dy^T H_s (columns s*F .. of the shared hidden)
            w.M = L.d;
            w.N = L.F;
            w.b_col0 = sh * L.F;
            w.C = gr->dW2;
            w.c_g0 = L.E + sh;
            w.c_gs = (long long)L.d * L.F;
            w.ldc = L.F;
            bwd(mDy, mHs, mDy, mHs, w, kBwdReduce, kEpiStore, tiles(w.M, w.N));
            BwdTcArgs a = f;  // dH_s = dy W2_s with the SwiGLU backward, in place
            a.N = L.F;
            a.K = L.d;
            a.b_g0 = L.E + sh;
            a.b_rows_per_group = L.d;
            a.C = const_cast<void*>(offset_elems(zs1, (size_t)sh * L.F, esz));
            a.C2 = const_cast<void*>(offset_elems(zs3, (size_t)sh * L.F, esz));
            a.e1 = a.C;
            a.e2 = a.C2;
            a.ldc = (long long)SF;
            bwd(kDy, mW2, kDy, mW2, a, kBwdRows, kEpiSwigluBwd, (long long)ceil_div(L.T, 128) * ceil_div(L.F, 256));
        }
        BwdTcArgs w = f;  // dW1_s = dZs1^T x, dW3_s = dZs3^T x
        w.M = (int)SF;
        w.N = L.d;
        w.C = gr->dW1;
        w.c_g0 = L.E;
        w.c_gs = (long long)L.F * L.d;
        w.ldc = L.d;
        bwd(mZs1, mX, mZs1, mX, w, kBwdReduce, kEpiStore, tiles(w.M, w.N));
        w.C = gr->dW3;
        bwd(mZs3, mX, mZs3, mX, w, kBwdReduce, kEpiStore, tiles(w.M, w.N));
        BwdTcArgs a = f;  // dXs = dZs1 W1_s + dZs3 W3_s
        a.N = L.d;
        a.K = (int)SF;
        a.b_g0 = L.E;
        a.b_rows_per_group = L.F;
        a.two_seg = 1;
        a.C = dxs;
        a.ldc = L.d;
        bwd(kZs1, mW1, kZs3, mW3, a, kBwdRows, kEpiStore, (long long)ceil_div(L.T, 128) * ceil_div(L.d, 256));
    }
    return e;
}

moe_status_t run_backward(Ctx& c, const void* dy, float d_aux, const moe_grads_t* gr)
{
    const Layout& L = c.L;
    if (L.T == 0) {  // an empty batch: every gradient is zero
        const size_t ES = (size_t)(L.E + L.S), w = ES * L.F * L.d * L.esz;
        const std::pair<void*, size_t> z[] = {{gr->dW_gate, 4ull * L.E * L.d}, {gr->db_gate, 4ull * L.E},
                                              {gr->dW1, w}, {gr->dW3, w}, {gr->dW2, w},
                                              {gr->db1, ES * L.F * L.esz}, {gr->db2, ES * L.d * L.esz},
                                              {gr->dW_noise, 4ull * L.E * L.d}, {gr->db_noise, 4ull * L.E}};
        for (const auto& q : z)
            if (q.first != nullptr && cudaMemsetAsync(q.first, 0, q.second, c.st) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const size_t esz = L.esz;
    const int types = c.bf16 ? kBwdTypesBf16 : kBwdTypesF32;
    const bool swiglu = c.p.act == MOE_ACT_SWIGLU, noisy = c.p.noisy_gating == 1;
    const float* logits = c.out->logits != nullptr ? c.out->logits : c.at<float>(L.off_logits);
    float* dgate = c.at<float>(L.off_bw_dgate);
    float* dl = c.at<float>(L.off_bw_dl);
    float* dn = noisy ? c.at<float>(L.off_bw_dn) : nullptr;
    float* dxr = c.at<float>(L.off_bw_dxr);
    void* dyp = c.at<void>(L.off_bw_dyp);
    void* z1 = c.at<void>(L.off_bw_z1);
    void* z3 = swiglu ? c.at<void>(L.off_bw_z3) : nullptr;
    const int* mtile = c.at<int>(L.off_mtile);
    const int* row_off = c.at<int>(L.off_row_off);
    const int* kept = c.at<int>(L.off_kept);
    const int32_t* slot_row = c.at<int32_t>(L.off_slot_row);
    const int mt_routed = L.rows_cap / kSegRows;
    auto grid_for = [&](long long tiles) { return (int)std::max(1ll, std::min(tiles, (long long)c.sms * 4)); };
    auto tiles = [](int M, int N) { return (long long)ceil_div(M, 128) * ceil_div(N, 64); };
    cudaError_t e = cudaSuccess;
    auto gemm = [&](const BwdGemmArgs& a, int ty, long long n_tiles) {
        if (e == cudaSuccess) e = launch_gemm_bwd_ffma(a, ty, grid_for(n_tiles), c.st, take_pdl(c));
    };
    auto colsum = [&](const ColsumArgs& a, int ty) {
        if (e == cudaSuccess) e = launch_colsum(a, ty, c.sms, c.st, take_pdl(c));
    };

    // combine: dYp = gate * dy on each kept slot's row, dgate = <dy, Yp>
    BwdCombineArgs cb{};
    cb.dy = dy;
    cb.yp = c.at<void>(L.off_yp);
    cb.dyp = dyp;
    cb.slot_row = slot_row;
    cb.gates = c.out->gates;
    cb.dgate = dgate;
    cb.T = L.T;
    cb.d = L.d;
    cb.k = L.k;
    e = launch_bwd_combine(cb, c.bf16, c.sms, c.st, take_pdl(c));

    // router: logit (and noise) gradients, then the router's weight and input gradients
    RouterBwdArgs rb{};
    rb.logits = logits;
    rb.idx = c.out->expert_idx;
    rb.dgate = dgate;
    rb.counts = c.out->counts;
    rb.d_aux = d_aux;
    rb.T = L.T;
    rb.E = L.E;
    rb.k = L.k;
    rb.renormalize = c.p.renormalize;
    rb.dl = dl;
    if (noisy) {
        rb.noise_parts = c.at<float>(L.off_nlogits);
        rb.k_splits = L.r_ksplits;
        rb.bn = c.in->b_noise;
        rb.eps = c.in->noise_eps;
        rb.dn = dn;
    }
    if (e == cudaSuccess) e = launch_router_bwd(rb, c.sms, c.st, take_pdl(c));
    if (L.tc_rbwd) {
        if (e == cudaSuccess) e = router_bwd_tc(c, dl, dn, dxr, gr);
    } else {
        {
            BwdGemmArgs a{};  // dW_gate[e, i] = sum_t dl[t, e] x[t, i]
            a.mode = kBwdFixed;
            a.epi = kEpiStore;
            a.A = dl;
            a.a_sm = 1;
            a.a_sk = L.E;
            a.B = c.in->x;
            a.b_sk = L.d;
            a.b_sn = 1;
            a.C = gr->dW_gate;
            a.c_sm = L.d;
            a.M = L.E;
            a.N = L.d;
            a.K = L.T;
            const int ty = c.bf16 ? kBwdTypesF32xBf16 : kBwdTypesF32;
            gemm(a, ty, tiles(a.M, a.N));
            if (noisy) {
                a.A = dn;
                a.C = gr->dW_noise;
                gemm(a, ty, tiles(a.M, a.N));
            }
            BwdGemmArgs r{};  // dx_router[t, i] = sum_e dl[t, e] W_gate[e, i] (+ dn W_noise)
            r.mode = kBwdFixed;
            r.epi = kEpiStore;
            r.A = dl;
            r.A2 = dn;
            r.a_sm = L.E;
            r.a_sk = 1;
            r.B = c.in->W_gate;
            r.B2 = noisy ? c.in->W_noise : nullptr;
            r.b_sk = L.d;
            r.b_sn = 1;
            r.C = dxr;
            r.c_sm = L.d;
            r.M = L.T;
            r.N = L.d;
            r.K = L.E;
            gemm(r, kBwdTypesF32, tiles(r.M, r.N));
        }
    }
    {
        ColsumArgs s{};
        s.lda = L.E;
        s.fixed_rows = L.T;
        s.G = 1;
        s.N = L.E;
        if (gr->db_gate) {
            s.A = dl;
            s.out = gr->db_gate;
            colsum(s, kBwdTypesF32);
        }
        if (gr->db_noise) {
            s.A = dn;
            s.out = gr->db_noise;
            colsum(s, kBwdTypesF32);
        }
    }

    void* dxs = L.S > 0 ? c.at<void>(L.off_bw_dxs) : nullptr;
    if (c.use_tc) {
        if (e == cudaSuccess) e = experts_bwd_tc(c, dy, gr);
    } else {
        // routed experts
        BwdGemmArgs rows{};  // row-grouped products over the expert segments
        rows.mode = kBwdRows;
        rows.mtile_off = mtile;
        rows.row_off = row_off;
        rows.rows = kept;
        rows.G = L.E;
        BwdGemmArgs red = rows;  // products reduced over the rows of each segment
        red.mode = kBwdReduce;
        const long long mt_tiles = mt_routed;
        if (c.p.act != MOE_ACT_RELU) {  // recompute the pre-activations z1 (+ b1) and z3
            BwdGemmArgs a = rows;
            a.epi = kEpiStore;
            a.A = c.at<void>(L.off_xp);
            a.a_sm = L.d;
            a.a_sk = 1;
            a.B = c.in->W1;
            a.b_sk = 1;
            a.b_sn = L.d;
            a.b_gs = (long long)L.F * L.d;
            a.C = z1;
            a.c_sm = L.F;
            a.bias = c.in->b1;
            a.N = L.F;
            a.K = L.d;
            gemm(a, types, mt_tiles * ceil_div(a.N, 64));
            if (swiglu) {
                a.B = c.in->W3;
                a.C = z3;
                a.bias = nullptr;
                gemm(a, types, mt_tiles * ceil_div(a.N, 64));
            }
        }
        {
            BwdGemmArgs a = red;  // dW2_e = dYp_e^T H_e
            a.epi = kEpiStore;
            a.A = dyp;
            a.a_sm = 1;
            a.a_sk = L.d;
            a.B = c.at<void>(L.off_h);
            a.b_sk = L.F;
            a.b_sn = 1;
            a.C = gr->dW2;
            a.c_gs = (long long)L.d * L.F;
            a.c_sm = L.F;
            a.M = L.d;
            a.N = L.F;
            gemm(a, types, L.E * tiles(a.M, a.N));
        }
        if (gr->db2) {
            ColsumArgs s{};
            s.A = dyp;
            s.lda = L.d;
            s.row_off = row_off;
            s.rows = kept;
            s.G = L.E;
            s.N = L.d;
            s.out = gr->db2;
            colsum(s, types);
        }
        {
            BwdGemmArgs a = rows;  // dH = dYp W2_e, then the activation backward
            a.A = dyp;
            a.a_sm = L.d;
            a.a_sk = 1;
            a.B = c.in->W2;
            a.b_sk = L.F;
            a.b_sn = 1;
            a.b_gs = (long long)L.d * L.F;
            a.C = z1;
            a.c_sm = L.F;
            a.N = L.F;
            a.K = L.d;
            if (c.p.act == MOE_ACT_RELU) {
                a.epi = kEpiReluBwd;
                a.e1 = c.at<void>(L.off_h);
            } else if (swiglu) {
                a.epi = kEpiSwigluBwd;
                a.e1 = z1;
                a.e2 = z3;
                a.C2 = z3;
            } else {
                a.epi = c.p.act == MOE_ACT_GELU_TANH ? kEpiGeluTanhBwd : kEpiGeluErfBwd;
                a.e1 = z1;
            }
            gemm(a, types, mt_tiles * ceil_div(a.N, 64));
        }
        {
            BwdGemmArgs a = red;  // dW1_e = dZ1_e^T Xp_e (and dW3_e from dZ3)
            a.epi = kEpiStore;
            a.A = z1;
            a.a_sm = 1;
            a.a_sk = L.F;
            a.B = c.at<void>(L.off_xp);
            a.b_sk = L.d;
            a.b_sn = 1;
            a.C = gr->dW1;
            a.c_gs = (long long)L.F * L.d;
            a.c_sm = L.d;
            a.M = L.F;
            a.N = L.d;
            gemm(a, types, L.E * tiles(a.M, a.N));
            if (swiglu) {
                a.A = z3;
                a.C = gr->dW3;
                gemm(a, types, L.E * tiles(a.M, a.N));
            }
        }
        if (gr->db1) {
            ColsumArgs s{};
            s.A = z1;
            s.lda = L.F;
            s.row_off = row_off;
            s.rows = kept;
            s.G = L.E;
            s.N = L.F;
            s.out = gr->db1;
            colsum(s, types);
        }
        {
            BwdGemmArgs a = rows;  // dXp = dZ1 W1_e (+ dZ3 W3_e), into the dYp buffer
            a.epi = kEpiStore;
            a.A = z1;
            a.A2 = z3;
            a.a_sm = L.F;
            a.a_sk = 1;
            a.B = c.in->W1;
            a.B2 = swiglu ? c.in->W3 : nullptr;
            a.b_sk = L.d;
            a.b_sn = 1;
            a.b_gs = (long long)L.F * L.d;
            a.C = dyp;
            a.c_sm = L.d;
            a.N = L.d;
            a.K = L.F;
            gemm(a, types, mt_tiles * ceil_div(a.N, 64));
        }

        // shared experts: gate 1 on every token (SwiGLU), hidden S*F, dO = dy
        if (L.S > 0) {
            void* zs1 = c.at<void>(L.off_bw_zs1);
            void* zs3 = c.at<void>(L.off_bw_zs3);
            const long long SF = (long long)L.S * L.F;
            BwdGemmArgs a{};
            a.mode = kBwdFixed;
            a.epi = kEpiStore;
            a.A = c.in->x;  // z = x W^T over the S*F concatenated rows
            a.a_sm = L.d;
            a.a_sk = 1;
            a.B = c.in->W1;
            a.b_sk = 1;
            a.b_sn = L.d;
            a.b_gs = (long long)L.F * L.d;
            a.b_g0 = L.E;
            a.C = zs1;
            a.c_sm = SF;
            a.M = L.T;
            a.N = (int)SF;
            a.K = L.d;
            gemm(a, types, tiles(a.M, a.N));
            a.B = c.in->W3;
            a.C = zs3;
            gemm(a, types, tiles(a.M, a.N));
            for (int sh = 0; sh < L.S; ++sh) {
                BwdGemmArgs b{};  // dH_s = dy W2_s with the SwiGLU backward, on columns s*F ..
                b.mode = kBwdFixed;
                b.epi = kEpiSwigluBwd;
                b.A = dy;
                b.a_sm = L.d;
                b.a_sk = 1;
                b.B = c.in->W2;
                b.b_sk = L.F;
                b.b_sn = 1;
                b.b_gs = (long long)L.d * L.F;
                b.b_g0 = L.E + sh;
                b.C = const_cast<void*>(offset_elems(zs1, (size_t)sh * L.F, esz));
                b.C2 = const_cast<void*>(offset_elems(zs3, (size_t)sh * L.F, esz));
                b.e1 = b.C;
                b.e2 = b.C2;
                b.c_sm = SF;
                b.M = L.T;
                b.N = L.F;
                b.K = L.d;
                // dW2_s = dy^T H_s first (it reads H_s, which the SwiGLU backward leaves alone)
                BwdGemmArgs w{};
                w.mode = kBwdFixed;
                w.epi = kEpiStore;
                w.A = dy;
                w.a_sm = 1;
                w.a_sk = L.d;
                w.B = offset_elems(c.at<void>(L.off_hs), (size_t)sh * L.F, esz);
                w.b_sk = SF;
                w.b_sn = 1;
                w.C = const_cast<void*>(offset_elems(gr->dW2, (size_t)(L.E + sh) * L.d * L.F, esz));
                w.c_sm = L.F;
                w.M = L.d;
                w.N = L.F;
                w.K = L.T;
                gemm(w, types, tiles(w.M, w.N));
                gemm(b, types, tiles(b.M, b.N));
            }
            BwdGemmArgs w{};  // dW1_s = dZs1^T x, dW3_s = dZs3^T x over the S*F rows
            w.mode = kBwdFixed;
            w.epi = kEpiStore;
            w.A = zs1;
            w.a_sm = 1;
            w.a_sk = SF;
            w.B = c.in->x;
            w.b_sk = L.d;
            w.b_sn = 1;
            w.C = const_cast<void*>(offset_elems(gr->dW1, (size_t)L.E * L.F * L.d, esz));
            w.c_sm = L.d;
            w.M = (int)SF;
            w.N = L.d;
            w.K = L.T;
            gemm(w, types, tiles(w.M, w.N));
            w.A = zs3;
            w.C = const_cast<void*>(offset_elems(gr->dW3, (size_t)L.E * L.F * L.d, esz));
            gemm(w, types, tiles(w.M, w.N));
            BwdGemmArgs x{};  // dXs = dZs1 W1_s + dZs3 W3_s
            x.mode = kBwdFixed;
            x.epi = kEpiStore;
            x.A = zs1;
            x.A2 = zs3;
            x.a_sm = SF;
            x.a_sk = 1;
            x.B = c.in->W1;
            x.B2 = c.in->W3;
            x.b_sk = L.d;
            x.b_sn = 1;
            x.b_gs = (long long)L.F * L.d;
            x.b_g0 = L.E;
            x.C = dxs;
            x.c_sm = L.d;
            x.M = L.T;
            x.N = L.d;
            x.K = (int)SF;
            gemm(x, types, tiles(x.M, x.N));
        }

    }

    BwdUnpermuteArgs u{};
    u.dy = dy;
    u.dxp = dyp;
    u.dxs = dxs;
    u.dxr = dxr;
    u.slot_row = slot_row;
    u.T = L.T;
    u.d = L.d;
    u.k = L.k;
    u.residual_mode = c.p.residual_mode;
    u.dx = gr->dx;
    if (e == cudaSuccess) e = launch_bwd_unpermute(u, c.bf16, c.sms, c.st, take_pdl(c));
    return cuda_status(e);
}

}  // namespace host
}  // namespace moe

using namespace moe;
using namespace moe::host;

extern "C" {

moe_status_t moe_workspace_size(const moe_params_t* params, size_t* bytes)
{
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t s = validate_params(params);
    if (s != MOE_OK) return s;
    *bytes = make_layout(*params).total;
    return MOE_OK;
}

moe_status_t moe_router_weights_size(const moe_params_t* params, size_t* bytes)
{
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t s = validate_params(params);
    if (s != MOE_OK) return s;
    if (params->dtype != MOE_BF16 || (params->flags & MOE_FLAG_FFMA_ROUTER)) return MOE_ERR_UNSUPPORTED;
    *bytes = 3 * sizeof(uint16_t) * (size_t)router_split_rows(params->E) * params->d_model *
             (params->noisy_gating == 1 ? 2 : 1);
    return MOE_OK;
}

moe_status_t moe_prepare_router_weights(const moe_params_t* params, const float* W_gate, const float* W_noise,
                                        void* prepared, size_t prepared_bytes, void* stream)
{
    size_t need = 0;
    moe_status_t s = moe_router_weights_size(params, &need);
    if (s != MOE_OK) return s;
    if (W_gate == nullptr || prepared == nullptr || !aligned16(prepared) || !aligned16(W_gate) ||
        (params->noisy_gating == 1) != (W_noise != nullptr) || (W_noise && !aligned16(W_noise)))
        return MOE_ERR_INVALID_ARG;
    if (prepared_bytes < need) return MOE_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_split_wgate(W_gate, params->E, params->d_model, prepared, sms, st, false);
    if (e == cudaSuccess && W_noise != nullptr)
        e = launch_split_wgate(W_noise, params->E, params->d_model, static_cast<char*>(prepared) + need / 2, sms, st,
                               false);
    return cuda_status(e);
}

moe_status_t moe_forward(const moe_params_t* params, const moe_inputs_t* inputs, moe_outputs_t* outputs,
                         void* workspace, size_t workspace_bytes, void* stream)
{
    return run_stages(params, inputs, outputs, workspace, workspace_bytes, stream,
                      {stage_router, stage_dispatch, stage_gemm, stage_combine});
}

moe_status_t moe_router(const moe_params_t* params, const moe_inputs_t* inputs, moe_outputs_t* outputs,
                        void* workspace, size_t workspace_bytes, void* stream)
{
    return run_stages(params, inputs, outputs, workspace, workspace_bytes, stream, {stage_router});
}

moe_status_t moe_dispatch(const moe_params_t* params, const moe_inputs_t* inputs, moe_outputs_t* outputs,
                          void* workspace, size_t workspace_bytes, void* stream)
{
    return run_stages(params, inputs, outputs, workspace, workspace_bytes, stream, {stage_dispatch});
}

moe_status_t moe_grouped_gemm(const moe_params_t* params, const moe_inputs_t* inputs, moe_outputs_t* outputs,
                              void* workspace, size_t workspace_bytes, void* stream)
{
    return run_stages(params, inputs, outputs, workspace, workspace_bytes, stream, {stage_gemm});
}

moe_status_t moe_combine(const moe_params_t* params, const moe_inputs_t* inputs, moe_outputs_t* outputs,
                         void* workspace, size_t workspace_bytes, void* stream)
{
    return run_stages(params, inputs, outputs, workspace, workspace_bytes, stream, {stage_combine});
}

moe_status_t moe_backward(const moe_params_t* params, const moe_inputs_t* inputs, const moe_outputs_t* outputs,
                          const void* dy, float d_aux, const moe_grads_t* grads, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    moe_status_t s = validate_params(params);
    if (s != MOE_OK) return s;
    if (!(params->flags & MOE_FLAG_TRAINING) || outputs == nullptr || inputs == nullptr) return MOE_ERR_INVALID_ARG;
    s = validate_grads(*params, inputs, dy, d_aux, grads);
    if (s != MOE_OK) return s;
    moe_outputs_t out = *outputs;  // read only
    Ctx c;
    s = prepare(params, inputs, &out, workspace, workspace_bytes, stream, c);
    if (s != MOE_OK) return s;
    return run_backward(c, dy, d_aux, grads);
}

moe_status_t moe_last_device_status(void* workspace, size_t workspace_bytes, void* stream)
{
    if (workspace == nullptr || workspace_bytes < sizeof(uint32_t)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_ERR_DEVICE_TIMEOUT;
    }
    return MOE_OK;
}

uint64_t moe_kernel_launches(void) { return moe::launch_counter().load(std::memory_order_relaxed); }

moe_status_t moe_check_bounded_wait(void* workspace, size_t workspace_bytes, uint32_t timeout_us, void* stream)
{
    if (workspace == nullptr || workspace_bytes < sizeof(uint32_t) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MOE_ERR_WORKSPACE;
    if (timeout_us < 1 || timeout_us > 1000000) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_wait_expires(static_cast<uint32_t*>(workspace), 1000ull * timeout_us,
                                           static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quantize_int4(const void* w, int32_t dtype, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                               void* stream)
{
    if (w == nullptr || q == nullptr || scale == nullptr || rows < 0 || cols < 1) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
    if (cols % MOE_INT4_GROUP != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    const int sms = sm_count();
    if (sms <= 0) return MOE_ERR_CUDA;
    return cuda_status(launch_quantize_int4(w, dtype == MOE_BF16, rows, cols, q, scale, sms,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quantize_int8(const void* w, int32_t dtype, int64_t rows, int32_t cols, int8_t* q, float* scale,
                               void* stream)
{
    if (w == nullptr || q == nullptr || scale == nullptr || rows < 0 || cols < 1) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    const int sms = sm_count();
    if (sms <= 0) return MOE_ERR_CUDA;
    return cuda_status(launch_quantize_int8(w, dtype == MOE_BF16, rows, cols, q, scale, sms,
                                            static_cast<cudaStream_t>(stream)));
}

const char* moe_status_string(moe_status_t status)
{
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    }
    return "MOE_ERR_UNKNOWN";
}

}  // extern "C"
