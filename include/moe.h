/*
 * moe.h -- C ABI of the B300 sparse Mixture-of-Experts FFN forward library
 * (libmoe_b300.so, sm_103a).
 *
 * The library computes, on one GPU, the forward pass of a sparse MoE FFN layer:
 * a softmax router over E experts, top-k selection with optional capacity and
 * residual pass-through, dispatch of tokens into expert-contiguous buffers, the
 * per-expert FFNs (plus always-on shared experts), the gate-weighted combine,
 * and the Switch load-balancing statistic N * sum_i f_i * P_i.
 *
 * Sources (web pages; cited by title and section):
 *   [Intro]  "混合专家模型MoE入门实战：从零搭建可运行的小型MoE模型" (0539edu.com/news/5495887)
 *   [Arch]   "MoE架构解析：混合专家模型原理与工程实践" (jsqmd.com/news/1258680)
 *   [Sparse] "MoE混合专家模型原理与实战：稀疏激活如何实现万亿参数高效推理" (framerc.cn/news/2939593)
 *   [Basic]  "混合专家 MOE 是什么" (dgblog.top/posts/ai/moe)
 *   [Switch] "MoE 混合专家模型串讲：从 Switch Transformer 到 DeepSeekMoE" (uestc.de5.net/blog/mixture-of-experts)
 *
 * Conventions shared by every entry point
 *   - All tensors are row-major and owned by the caller.  Pointers in
 *     moe_inputs_t / moe_outputs_t and the workspace are DEVICE pointers of the
 *     current CUDA device; every one must be 16-byte aligned.
 *   - Weights use the nn.Linear [out, in] layout: W1/W3 are [E+S, d_ff, d_model],
 *     W2 is [E+S, d_model, d_ff]; the E routed experts come first, the S shared
 *     experts last.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every entry
 *     point only enqueues work on it: no allocation, no host synchronisation
 *     (moe_last_device_status excepted), no global state.  A workspace may be
 *     used by one stream at a time.
 *   - Validation happens before any launch.  On a non-OK status nothing was
 *     enqueued.  Asynchronous device faults surface at the caller's next
 *     synchronisation as usual.
 *   - For an empty batch (T == 0) the arrays with T rows may be NULL.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad sizes, null or unaligned pointers, k > E ... */
    MOE_ERR_UNSUPPORTED = 2,   /* a valid combination this build does not implement */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_size */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = 5 /* a bounded device wait expired (moe_last_device_status) */
} moe_status_t;

typedef enum {
    MOE_ACT_RELU = 0,      /* max(z, 0) */
    MOE_ACT_GELU_TANH = 1, /* 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) */
    MOE_ACT_GELU_ERF = 2,  /* 0.5 z (1 + erf(z / sqrt 2)) */
    MOE_ACT_SWIGLU = 3     /* W2 (silu(W1 x) * (W3 x)); no biases */
} moe_act_t;

typedef enum {
    MOE_F32 = 0, /* x, expert weights, biases and y in fp32 (CUDA-core FFMA experts) */
    MOE_BF16 = 1 /* x, expert weights, biases and y in bf16 (tensor-core experts) */
} moe_dtype_t;

/* moe_params_t.flags */
#define MOE_FLAG_FFMA_EXPERTS 1u /* run bf16 experts on the CUDA-core FFMA grouped GEMM
                                    (cross-check kernel) instead of the tcgen05 one */
#define MOE_FLAG_FFMA_ROUTER 2u  /* compute bf16 router logits with CUDA-core FFMA
                                    (cross-check kernel) instead of the tensor-core
                                    three-term split; fp32 layers always use FFMA */
#define MOE_FLAG_UNFUSED_EXPERTS 4u /* run the routed experts' two layers as two
                                       grouped-GEMM launches instead of one fused
                                       persistent launch (cross-check path) */
#define MOE_FLAG_TRAINING 8u /* the workspace also holds what moe_backward needs (the
                                forward keeps the router logits; backward buffers are
                                reserved); required by moe_backward */

/* Limits of this build. */
#define MOE_MAX_EXPERTS 512 /* E (routed) */
#define MOE_MAX_TOPK 32     /* k */

typedef struct {
    int32_t T;          /* tokens (rows of x) >= 0; T == 0 (an empty batch) launches no kernel:
                           the forward writes counts = 0 and aux = 0, the backward zero gradients */
    int32_t d_model;    /* d, multiple of 8 */
    int32_t d_ff;       /* F, hidden width of one expert, multiple of 8 */
    int32_t E;          /* routed experts, 1..MOE_MAX_EXPERTS */
    int32_t k;          /* experts per token, 1..min(E, MOE_MAX_TOPK) */
    int32_t n_shared;   /* S always-on shared experts (gate 1); SwiGLU only */
    float capacity_factor; /* <= 0: no limit; else C = floor(T * cf / E) rows per expert */
    int32_t renormalize;   /* 1: gates = p / sum of the k selected p; 0: gates = p */
    int32_t residual_mode; /* 0: y = x added only to tokens whose routed slots were all
                              dropped; 1: y += x for every token */
    int32_t act;        /* moe_act_t */
    int32_t dtype;      /* moe_dtype_t */
    uint32_t flags;     /* MOE_FLAG_* */
    int32_t noisy_gating;  /* 1: noisy top-k gating (training mode, see below); 0: off */
    float noise_min_std;   /* floor added to the noise scale; >= 0, finite */
    int32_t weight_format; /* moe_weight_format_t */
} moe_params_t;

/* Expert weight storage ([Arch] §"部署实践": 8-bit expert weights; [Sparse]
 * §"量化与PagedAttention结合": experts quantised, router kept precise).
 * MOE_WEIGHTS_INT8: W1, W3, W2 hold int8 q with one fp32 scale per output row,
 * W[e, n, :] = q[e, n, :] * scale[e, n] (moe_quantize_int8 makes them).  Needs
 * dtype == MOE_BF16, the tensor-core expert path, n_shared == 0, no
 * MOE_FLAG_TRAINING, and d_model and d_ff multiples of 16; otherwise
 * MOE_ERR_UNSUPPORTED.  The router weights stay fp32. */
typedef enum {
    MOE_WEIGHTS_DTYPE = 0, /* expert weights in the layer dtype */
    MOE_WEIGHTS_INT8 = 1,  /* int8 expert weights + fp32 per-row scales */
    MOE_WEIGHTS_INT4 = 2   /* 4-bit expert weights + fp32 scales per group of MOE_INT4_GROUP inputs */
} moe_weight_format_t;

/* MOE_WEIGHTS_INT4 ([Sparse] §"量化与PagedAttention结合": the experts alone
 * quantised to INT4 with AWQ, whose storage is group-wise): W[e, n, c] =
 * q[e, n, c] * scale[e, n, c / MOE_INT4_GROUP] with q in [-7, 7]; two values per
 * byte, column 2i in the low nibble and 2i + 1 in the high nibble (4-bit two's
 * complement), so W1 and W3 are [E, F, d / 2] bytes and W2 is [E, d, F / 2];
 * W1_scale and W3_scale are [E, F, d / MOE_INT4_GROUP] fp32, W2_scale
 * [E, d, F / MOE_INT4_GROUP] (moe_quantize_int4 makes them).  Needs dtype ==
 * MOE_BF16, n_shared == 0, no MOE_FLAG_TRAINING or MOE_FLAG_FFMA_EXPERTS, and
 * d_model and d_ff multiples of MOE_INT4_GROUP; otherwise MOE_ERR_UNSUPPORTED.
 * The tensor core multiplies bf16 activations by the weights dequantised to bf16
 * (q * scale in fp32, rounded once). */
#define MOE_INT4_GROUP 128

/* Noisy top-k gating ([Arch] §2.1 noisy_top_k_gating; [Switch] §"代码实战"
 * NoisyTop1Gate).  With noisy_gating = 1 the router also computes
 *     noise_logits[t,e] = sum_i x[t,i] W_noise[e,i] + b_noise[e]     (fp32)
 * and replaces the logits by
 *     logits[t,e] + noise_eps[t,e] * (softplus(noise_logits[t,e]) + noise_min_std)
 * before softmax, top-k, gates and the balance statistic, which therefore all
 * see the noisy logits (outputs.logits holds them too).  noise_eps is a [T,E]
 * array of standard normal draws supplied by the caller: the library draws no
 * random numbers, so a forward is a deterministic function of its inputs.
 * noise_min_std = 0 is the [Arch] form, 1e-2 the [Switch] one.  With
 * noisy_gating = 0, W_noise, b_noise and noise_eps must be NULL. */

typedef struct {
    const void* x;       /* [T, d] dtype */
    const float* W_gate; /* [E, d] fp32 router weights */
    const float* b_gate; /* [E] fp32 router bias, or NULL */
    const void* W1;      /* [E+S, F, d] dtype */
    const void* W3;      /* [E+S, F, d] dtype; required iff act == SWIGLU, else NULL */
    const void* W2;      /* [E+S, d, F] dtype */
    const void* b1;      /* [E+S, F] dtype or NULL (must be NULL for SwiGLU) */
    const void* b2;      /* [E+S, d] dtype or NULL (must be NULL for SwiGLU) */
    const float* W_noise;   /* [E, d] fp32 noise projection; required iff noisy_gating */
    const float* b_noise;   /* [E] fp32 noise projection bias, or NULL */
    const float* noise_eps; /* [T, E] fp32 standard normal draws; required iff noisy_gating */
    const float* W1_scale;  /* INT8: [E, F]; INT4: [E, F, d / MOE_INT4_GROUP]; fp32; required iff
                               weight_format != MOE_WEIGHTS_DTYPE, else NULL */
    const float* W3_scale;  /* the same shape; iff quantised and SwiGLU */
    const float* W2_scale;  /* INT8: [E, d]; INT4: [E, d, F / MOE_INT4_GROUP]; iff quantised */
    const void* router_weights; /* the router weights as moe_prepare_router_weights made them from
                                   W_gate (and W_noise) for these params, or NULL: the router then
                                   makes them in the workspace on every call.  Only for layers
                                   whose router runs on the tensor core (bf16, no
                                   MOE_FLAG_FFMA_ROUTER); otherwise it must be NULL */
} moe_inputs_t;

typedef struct {
    void* y;             /* [T, d] dtype: the layer output */
    int32_t* expert_idx; /* [T, k] selected experts, by router logit descending, ties to
                            the lower index */
    float* gates;        /* [T, k] fp32 gate of each slot (before drops) */
    int32_t* counts;     /* [E] tokens routed to each expert before capacity drops */
    uint8_t* dropped;    /* [T, k] 1 = slot dropped by the capacity limit */
    float* aux;          /* [1] E * sum_e (counts_e / (T k)) * (mean_t p[t,e]) */
    float* logits;       /* [T, E] fp32 router logits (the noisy ones under noisy gating),
                            or NULL (not written) */
    float* probs;        /* [T, E] fp32 router probabilities, or NULL */
    int32_t* perm_row;   /* [T, k] row of the slot in the expert-contiguous, token-ascending,
                            unpadded order of kept slots; -1 if dropped; or NULL */
} moe_outputs_t;

/* Router weights prepared once per weight update.  The tensor-core router of bf16
 * layers multiplies x by W_gate split exactly into three bf16 terms
 * (W = hi + mid + lo; [Switch] §"选择性精度" asks for an fp32 router); by default
 * every call makes that split in its workspace (one small kernel).  A caller whose
 * router weights change only at weight updates can make it once:
 * moe_router_weights_size gives the bytes (it depends on E, d_model and
 * noisy_gating only), moe_prepare_router_weights writes the split of W_gate (and,
 * with noisy gating, of W_noise) into a caller-owned, 16-byte aligned device
 * buffer on `stream`, and moe_inputs_t.router_weights points the layer at it.  The
 * buffer is valid for any T.  Layers whose router runs on CUDA cores (fp32, or
 * MOE_FLAG_FFMA_ROUTER) return MOE_ERR_UNSUPPORTED. */
moe_status_t moe_router_weights_size(const moe_params_t* params, size_t* bytes);
moe_status_t moe_prepare_router_weights(const moe_params_t* params, const float* W_gate, const float* W_noise,
                                        void* prepared, size_t prepared_bytes, void* stream);

/* Bytes of device workspace moe_forward needs for these params.  Depends only
 * on the params.  The workspace must be 256-byte aligned and must be zeroed
 * once before its first use (the library keeps it consistent afterwards). */
moe_status_t moe_workspace_size(const moe_params_t* params, size_t* bytes);

/* The whole layer: moe_router, moe_dispatch, moe_grouped_gemm, moe_combine in
 * that order on `stream`.  Writes every output of moe_outputs_t. */
moe_status_t moe_forward(const moe_params_t* params, const moe_inputs_t* inputs,
                         moe_outputs_t* outputs, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Stage 1, router.  logits[t,e] = sum_i x[t,i] W_gate[e,i] + b_gate[e] in fp32
 * ([Basic] §"公式：三步走"; the router runs in fp32 as [Switch] §"选择性精度"
 * prescribes), p = softmax over the E routed experts ([Basic] §"一个小算例"),
 * the k largest logits per token (warp-reduction top-k; [Intro] §3.3, [Arch]
 * §2.1), gates = p or p renormalised over the k ([Intro] §3.3), and per-block
 * column sums of p for the balance statistic.  Writes expert_idx, gates and the
 * optional logits/probs; the rest lives in the workspace. */
moe_status_t moe_router(const moe_params_t* params, const moe_inputs_t* inputs,
                        moe_outputs_t* outputs, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Stage 2, dispatch.  Per-expert histogram in shared memory and a device-wide
 * scan over token chunks give counts and token-order positions; capacity
 * C = floor(T cf / E) ([Arch] §3.1 expert_capacity, [Switch] §"专家容量")
 * drops the slots at position >= C; every kept token row is copied (16-byte
 * vectors) into an expert-contiguous buffer whose expert segments are padded
 * to 128 rows ([Intro] §2.4 scatter-gather).  Also computes the balance
 * statistic ([Intro] §3.4, [Switch] §"负载均衡损失函数").  Writes counts,
 * dropped, aux and perm_row.  Requires moe_router on the same workspace. */
moe_status_t moe_dispatch(const moe_params_t* params, const moe_inputs_t* inputs,
                          moe_outputs_t* outputs, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Stage 3, experts.  For every expert segment, H = act(Xp W1^T + b1) or SwiGLU
 * silu(Xp W1^T) * (Xp W3^T), then Yp = H W2^T + b2 ([Intro] §3.2, [Sparse]
 * §3.1); shared experts run on all T tokens as one SwiGLU of hidden S*d_ff
 * ([Switch] §"共享专家隔离").  bf16: tcgen05/TMEM grouped GEMM fed by TMA;
 * fp32: CUDA-core FFMA grouped GEMM.  Results stay in the workspace.
 * Requires moe_dispatch on the same workspace. */
moe_status_t moe_grouped_gemm(const moe_params_t* params, const moe_inputs_t* inputs,
                              moe_outputs_t* outputs, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Stage 4, combine.  y[t] = sum over kept slots of gate * expert output (fp32
 * accumulation, slot order) + shared output + x[t] when residual_mode says so
 * ([Intro] §3.4, [Basic] third formula, [Switch] §"专家容量": a dropped token
 * gets 0 + x = x).  Writes y.  Requires moe_grouped_gemm on the same workspace. */
moe_status_t moe_combine(const moe_params_t* params, const moe_inputs_t* inputs,
                         moe_outputs_t* outputs, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Gradients written by moe_backward (caller-owned device arrays, 16-byte aligned). */
typedef struct {
    void* dx;         /* [T, d] dtype */
    float* dW_gate;   /* [E, d] fp32 */
    float* db_gate;   /* [E] fp32; required iff inputs.b_gate != NULL, else NULL */
    void* dW1;        /* [E+S, F, d] dtype */
    void* dW3;        /* [E+S, F, d] dtype; required iff act == SWIGLU, else NULL */
    void* dW2;        /* [E+S, d, F] dtype */
    void* db1;        /* [E+S, F] dtype; required iff inputs.b1 != NULL, else NULL */
    void* db2;        /* [E+S, d] dtype; required iff inputs.b2 != NULL, else NULL */
    float* dW_noise;  /* [E, d] fp32; required iff noisy_gating, else NULL */
    float* db_noise;  /* [E] fp32; required iff noisy_gating and b_noise != NULL, else NULL */
} moe_grads_t;

/* Backward pass of the layer ([Intro] §3.4-§3.5 trains the layer end to end
 * with task loss + coef * aux loss; [Switch] §"负载均衡损失函数": P_i is
 * differentiable, f_i is not).  Given dy = dL/dy [T, d] (dtype, device) and
 * d_aux = dL/d aux (e.g. the aux-loss coefficient), writes every gradient of
 * moe_grads_t.  The forward's discrete decisions (top-k, capacity drops,
 * pass-through) are held fixed: the router receives gradient through the gate
 * values and P_i only.  Gate gradients pass through the renormalisation when it
 * applies; under noisy gating the noise projection receives
 * dL/dn = dL/dlogit * eps * sigmoid(n) (the draws are data).
 *
 * Requires MOE_FLAG_TRAINING in params.flags and, on the same workspace and
 * stream, a moe_forward with the same params, inputs and outputs whose results
 * are still in place (the backward reads expert_idx, gates, counts and the
 * optional logits from `outputs`, and the permuted activations, hidden
 * activations and expert outputs from the workspace).  Gradients are computed
 * in fp32 and rounded once to the destination type; weight gradients are
 * written (not accumulated).  Under MOE_FLAG_TRAINING the forward also keeps
 * the first layer's pre-activations in the workspace; the backward consumes
 * them (overwrites them with their gradients), so each moe_backward needs its
 * own preceding moe_forward.  Validation happens before any launch. */
moe_status_t moe_backward(const moe_params_t* params, const moe_inputs_t* inputs,
                          const moe_outputs_t* outputs, const void* dy, float d_aux,
                          const moe_grads_t* grads, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Expert parallelism over G ranks, emulated on this GPU ([Arch] §3.2
 * "分布式训练优化": experts placed on different devices, and the mixed data +
 * expert parallel mode in which the data is sharded over the workers, each
 * worker holds a part of the experts and tokens cross devices; [Arch] §5
 * (问题3): the exchange is an AllToAll; [Sparse] §4.2 "专家分片": 64 experts
 * cut over 4 cards).
 *
 * Rank r holds the tokens [floor(r T / G), floor((r+1) T / G)) and the experts
 * [r E/G, (r+1) E/G) (E must be a multiple of G).  Every rank routes its own
 * tokens, applies the capacity rule to its shard alone
 * (C_r = floor(T_r * cf / E), positions in the shard's token order), and sends
 * every kept slot's token row to the owner of its expert; each owner runs its
 * experts on the rows it received (its receive buffer holds its experts in
 * ascending order and, inside one expert, the rows of rank 0, 1, ... in token
 * order); the outputs travel back and every rank combines its own tokens
 * (shared experts: each rank on its own tokens).  Each rank has a private
 * region of the workspace; the only data that crosses ranks is moved by the
 * library's exchange kernels (a counts exchange, the token all-to-all and its
 * reverse), all on `stream`.
 *
 * The outputs are those of moe_forward, for the whole batch, with these
 * meanings: counts = every rank's slots per expert before drops (summed over
 * ranks); dropped = the per-shard capacity drops; aux = the balance statistic
 * reduced over all ranks (f and P over all T tokens); perm_row = the slot's row
 * in the concatenation of all ranks' receive buffers (rank 0's first,
 * unpadded), -1 if dropped.  Without a capacity limit the result is the single
 * rank layer's, and perm_row equals moe_forward's.
 *
 * Supported: the bf16 tensor-core experts (fused kernel) and the FFMA experts
 * (fp32, or MOE_FLAG_FFMA_EXPERTS); quantised weights, MOE_FLAG_UNFUSED_EXPERTS and
 * MOE_FLAG_TRAINING return MOE_ERR_UNSUPPORTED.  G outside 1..MOE_EP_MAX_RANKS
 * or E not a multiple of G returns MOE_ERR_INVALID_ARG.  The workspace
 * (moe_ep_workspace_size) must be zeroed once before its first use; bounded
 * device waits of every rank report to its first word (moe_last_device_status). */
#define MOE_EP_MAX_RANKS 16
moe_status_t moe_ep_workspace_size(const moe_params_t* params, int32_t G, size_t* bytes);
moe_status_t moe_forward_ep(const moe_params_t* params, int32_t G, const moe_inputs_t* inputs,
                            moe_outputs_t* outputs, void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, reads and clears the workspace's device error word.
 * Returns MOE_ERR_DEVICE_TIMEOUT if a bounded device wait expired since the last
 * call, MOE_ERR_CUDA if the synchronisation failed, else MOE_OK.  For tests and
 * debugging; not needed on the hot path. */
moe_status_t moe_last_device_status(void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free dispatch positions.  The pages have no counterpart: this is an
 * addition for callers that cannot allocate device memory when they route tokens
 * (an engine that owns all device memory through its own fixed pool and forbids
 * libraries from allocating, or a latency-critical path that cannot pay for
 * cudaMalloc's implicit synchronisation) and so cannot provide the workspace of
 * moe_workspace_size.
 *
 * From the router's expert_idx [T, k] (as moe_router writes it) computes what
 * moe_dispatch computes for the same selection: counts [E] (tokens per expert
 * before drops), dropped [T, k] (1 = over the capacity floor(T cf / E)) and
 * perm_row [T, k] (row in the expert-contiguous, token-ascending order of kept
 * slots, -1 if dropped).  It does not compute the balance statistic and does not
 * permute token rows.  Indices outside [0, E) are not counted and their slots are
 * reported as dropped.
 *
 * Scratch: a static device array of about 1 MB inside the library, one per device
 * that loads the library, held until the process exits.  Limits: T * k <=
 * MOE_NOALLOC_MAX_SLOTS and E <= MOE_MAX_EXPERTS; larger problems return
 * MOE_ERR_INVALID_ARG and enqueue nothing.  The first call on a device looks up
 * the array's device address (with that device current) and keeps it; make that
 * first call before starting any stream capture.  A lookup that fails returns
 * MOE_ERR_CUDA, enqueues nothing and is tried again by the next call.  Every call
 * clears the scan's arrival counter before its kernels run, and overwrites every
 * other scratch word it reads.  All calls on a device share the array:
 * calls whose work overlaps on the GPU (e.g. on two streams) race; calls ordered on
 * one stream are safe.  Allocates nothing; all pointers are device pointers. */
#define MOE_NOALLOC_MAX_SLOTS 131072
moe_status_t moe_dispatch_positions_noalloc(const moe_params_t* params,
                                            const int32_t* expert_idx, int32_t* counts,
                                            uint8_t* dropped, int32_t* perm_row, void* stream);

/* Number of kernels this library has launched in this process since it was
 * loaded, counting launches recorded into a CUDA graph under stream capture
 * (a graph replay launches no kernel through the library and counts nothing).
 * The difference across one call is the number of kernels that call enqueues.
 * Host-side counter; needs no device. */
uint64_t moe_kernel_launches(void);

/* Quantise `rows` rows of `cols` weights (device, `dtype` MOE_BF16 or MOE_F32,
 * row-major) to int8 with one scale per row: scale = max |w| / 127 (IEEE fp32),
 * q = round-half-even(w / scale) clamped to [-127, 127]; an all-zero row gets
 * scale 0 and q 0.  For a layer's W1, W3 ([E, F, d]) call it with rows = E*F,
 * cols = d; for W2 ([E, d, F]) with rows = E*d, cols = F.  Enqueues one kernel. */
moe_status_t moe_quantize_int8(const void* w, int32_t dtype, int64_t rows, int32_t cols, int8_t* q,
                               float* scale, void* stream);

/* Quantise `rows` rows of `cols` weights (device, `dtype` MOE_BF16 or MOE_F32,
 * row-major; cols a multiple of MOE_INT4_GROUP) to 4 bits with one scale per
 * group of MOE_INT4_GROUP consecutive columns: scale = max |w| / 7 over the group
 * (IEEE fp32), q = round-half-even(w / scale) clamped to [-7, 7]; an all-zero
 * group gets scale 0 and q 0.  Writes q packed two per byte ([rows, cols / 2],
 * column 2i in the low nibble) and scale [rows, cols / MOE_INT4_GROUP].  For a
 * layer's W1, W3 ([E, F, d]) call it with rows = E*F, cols = d; for W2
 * ([E, d, F]) with rows = E*d, cols = F.  Enqueues one kernel. */
moe_status_t moe_quantize_int4(const void* w, int32_t dtype, int64_t rows, int32_t cols, uint8_t* q,
                               float* scale, void* stream);

/* Diagnostic: enqueues one kernel whose bounded wait (on a barrier that nothing
 * arrives at) expires after timeout_us microseconds (1 .. 1e6) and records the
 * expiry in the workspace's error word, exactly as the layer's kernels do when a
 * wait of theirs expires.  The next moe_last_device_status on this workspace then
 * returns MOE_ERR_DEVICE_TIMEOUT (and clears the word); the CUDA context stays
 * usable.  For testing the failure-detection path; not needed otherwise. */
moe_status_t moe_check_bounded_wait(void* workspace, size_t workspace_bytes, uint32_t timeout_us,
                                    void* stream);

/* Static, human-readable name of a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
