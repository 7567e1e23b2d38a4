/*
 * moe_oracle.c -- plain fp64 CPU oracle for the forward pass of a sparse
 * Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA library: it is written from the
 * pages' definitions alone, as loops over tokens and experts, in double
 * precision, with no blocking, fusion or reordering.  Inputs are read in the
 * storage type the caller hands over (fp64, fp32 or bf16 bit patterns); every
 * arithmetic step is done in double.
 *
 * Sources (web pages; cited by title and section):
 *   [Intro]  "混合专家模型MoE入门实战：从零搭建可运行的小型MoE模型" (0539edu.com/news/5495887)
 *   [Arch]   "MoE架构解析：混合专家模型原理与工程实践" (jsqmd.com/news/1258680)
 *   [Sparse] "MoE混合专家模型原理与实战：稀疏激活如何实现万亿参数高效推理" (framerc.cn/news/2939593)
 *   [Basic]  "混合专家 MOE 是什么" (dgblog.top/posts/ai/moe)
 *   [Switch] "MoE 混合专家模型串讲：从 Switch Transformer 到 DeepSeekMoE" (uestc.de5.net/blog/mixture-of-experts)
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - top-k ties go to the lower expert index; slots are ordered by score descending;
 *   - capacity C = floor(T*cf/E) with no factor k; cf <= 0 means "no limit";
 *   - capacity priority is ascending token order (slot order inside a token cannot
 *     matter: a token never picks the same expert twice);
 *   - f_i counts the router's selection before capacity drops, normalised by T*k;
 *   - residual mode 0 adds x only to tokens whose routed slots were all dropped,
 *     mode 1 adds x to every token;
 *   - SwiGLU (absent from the pages) is W2 (silu(W1 x) * (W3 x)), silu(z) = z/(1+e^-z);
 *   - noisy gating: the noisy logits replace the clean ones in every later step
 *     (softmax, top-k, gates, balance statistic); the normal draws are an input.
 *
 * Every function here is pinned by CPU tests against values the pages print,
 * closed forms, invariants and brute force (tests/test_oracle_pins.py); the
 * backward pass against finite differences of the forward and the dense-MLP
 * special case (tests/test_oracle_backward_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Storage codes of the caller's arrays (decoding only). */
enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

/* Expert activation codes. */
enum { ORC_RELU = 0, ORC_GELU_TANH = 1, ORC_GELU_ERF = 2, ORC_SWIGLU = 3 };

/* Read element i of an array stored as fp64, fp32 or bf16, exactly, as a double. */
static double rd(const void* p, int code, size_t i)
{
    if (code == ORC_F64) return ((const double*)p)[i];
    if (code == ORC_F32) return (double)((const float*)p)[i];
    uint32_t u = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Expert capacity.  [Arch] §3.1 "容量因子": int(batch_size * capacity_factor /
 * num_experts); [Intro] §4.2 gives the worked number 1000 tokens, 8 experts,
 * factor 1.25 -> 156.  Returns -1 for "no capacity limit" (cf <= 0). */
long long orc_capacity(long long T, long long E, double cf)
{
    if (cf <= 0.0) return -1;
    return (long long)floor((double)T * cf / (double)E);
}

/* ------------------------------------------------------------------------ */
/* Step 1 -- router logits.  [Basic] §"公式：三步走" first formula: the router
 * is W_g x with W_g of shape experts x input dim; [Intro] §3.3 and [Switch]
 * §"从传统 MoE 到 Switch Routing" use the same linear router (with an optional
 * bias, as nn.Linear has).  logits[t,e] = sum_i x[t,i] * Wg[e,i] + bg[e]. */
void orc_router_logits(int T, int d, int E,
                       const void* x, int x_code,
                       const void* wg, int wg_code,
                       const void* bg, int bg_code,
                       double* logits)
{
    #pragma omp parallel for schedule(static)
    for (long t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int i = 0; i < d; ++i)
                s += rd(x, x_code, (size_t)t * d + i) * rd(wg, wg_code, (size_t)e * d + i);
            if (bg) s += rd(bg, bg_code, (size_t)e);
            logits[(size_t)t * E + e] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Step 1' -- noisy top-k gating (training mode).  [Arch] §2.1
 * noisy_top_k_gating: a second linear map of the token, x W_noise, passed
 * through softplus, scales a standard normal draw that is added to the clean
 * logits; the noisy logits then go through the same top-k gating.  [Switch]
 * §"代码实战" NoisyTop1Gate gives the same step with a bias on the noise
 * projection and a floor of 1e-2 added to the softplus (min_std below; 0 for
 * the [Arch] form), and feeds the noisy logits to softmax, argmax and the
 * balance statistic alike.  The normal draws are an input (eps, [T,E]).
 *   noisy[t,e] = clean[t,e] + eps[t,e] * (softplus(noise_logits[t,e]) + min_std)
 * softplus(z) = log(1 + e^z), evaluated as max(z,0) + log1p(e^-|z|), which is
 * the same number without overflow. */
double orc_softplus(double z)
{
    return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

void orc_noisy_logits(int T, int E, const double* clean, const double* noise_logits,
                      const void* eps, int eps_code, double min_std, double* noisy)
{
    for (size_t i = 0; i < (size_t)T * E; ++i)
        noisy[i] = clean[i] + rd(eps, eps_code, i) * (orc_softplus(noise_logits[i]) + min_std);
}

/* ------------------------------------------------------------------------ */
/* Step 2 -- softmax over the E routed experts.  [Basic] §"一个小算例":
 * softmax(z)_i = e^{z_i} / sum_j e^{z_j}.  The maximum is subtracted first;
 * that leaves every ratio unchanged. */
void orc_softmax(int T, int E, const double* logits, double* probs)
{
    #pragma omp parallel for schedule(static)
    for (long t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        double m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        double den = 0.0;
        for (int e = 0; e < E; ++e) den += exp(l[e] - m);
        for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = exp(l[e] - m) / den;
    }
}

/* ------------------------------------------------------------------------ */
/* Step 3 -- top-k selection.  [Intro] §3.3 (torch.topk on the softmax
 * weights), [Arch] §2.1 (top_k on the logits): softmax is monotone, so both
 * pick the same experts.  Slot j holds the j-th largest score; equal scores
 * go to the lower expert index. */
void orc_topk(int T, int E, int k, const double* scores, int32_t* idx)
{
    #pragma omp parallel
    {
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
        #pragma omp for schedule(static)
        for (long t = 0; t < T; ++t) {
            const double* s = scores + (size_t)t * E;
            memset(taken, 0, (size_t)E);
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || s[e] > s[best]) best = e;
                }
                taken[best] = 1;
                idx[(size_t)t * k + j] = best;
            }
        }
        free(taken);
    }
}

/* ------------------------------------------------------------------------ */
/* Step 4 -- gates.  The gate of slot j is the router probability of its
 * expert.  With renormalize != 0 the k gates are divided by their sum
 * ([Intro] §3.3, "重新归一化 Top-K 权重"); otherwise they are the raw
 * probabilities (Switch routing keeps p of the chosen expert, [Switch] §"门控
 * 网络与稀疏路由"; DeepSeekMoE sets g = s inside the top-K, [Switch]
 * §"数学定义"). */
void orc_gates(int T, int E, int k, const double* probs, const int32_t* idx,
               int renormalize, double* gates)
{
    for (long t = 0; t < T; ++t) {
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            double g = probs[(size_t)t * E + idx[(size_t)t * k + j]];
            gates[(size_t)t * k + j] = g;
            sum += g;
        }
        if (renormalize)
            for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] /= sum;
    }
}

/* ------------------------------------------------------------------------ */
/* Steps 5-6 -- routed counts and capacity in token order.
 * counts[e] = number of (t, j) with idx[t,j] == e, before any drop ([Intro]
 * §3.4, the one_hot frequency).  Walking tokens in ascending order, the slot
 * (t, j) gets position pos = number of earlier tokens routed to the same
 * expert; it is kept iff C < 0 or pos < C.  A token over capacity skips the
 * expert ([Switch] §"专家容量": f(x) = 0 for dropped tokens).
 * perm_row is the slot's row in the expert-contiguous, token-ascending,
 * unpadded order (offset of the expert's kept rows + pos), -1 if dropped. */
void orc_dispatch(int T, int E, int k, const int32_t* idx, long long C,
                  int32_t* counts, int32_t* pos, uint8_t* dropped, int32_t* perm_row)
{
    long long* seen = (long long*)calloc((size_t)E, sizeof(long long));
    long long* start = (long long*)calloc((size_t)E + 1, sizeof(long long));
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            size_t s = (size_t)t * k + j;
            int e = idx[s];
            counts[e] += 1;
            long long p = seen[e]++;
            pos[s] = (int32_t)p;
            dropped[s] = (uint8_t)(C >= 0 && p >= C);
        }
    }
    for (int e = 0; e < E; ++e) {
        long long kept = counts[e];
        if (C >= 0 && kept > C) kept = C;
        start[e + 1] = start[e] + kept;
    }
    for (size_t s = 0; s < (size_t)T * k; ++s)
        perm_row[s] = dropped[s] ? -1 : (int32_t)(start[idx[s]] + pos[s]);
    free(seen);
    free(start);
}

/* ------------------------------------------------------------------------ */
/* Switch load-balancing statistic N * sum_i f_i * P_i.  [Intro] §3.4 (code and
 * text: equals about 1 when balanced, larger when not), [Switch]
 * §"负载均衡损失函数" (f_i hard assignment fraction, P_i mean router
 * probability; f = P = 1/N gives the minimum).  f_i = counts_i / (T*k). */
double orc_aux(int T, int E, int k, const int32_t* counts, const double* probs)
{
    double aux = 0.0;
    for (int e = 0; e < E; ++e) {
        double P = 0.0;
        for (long t = 0; t < T; ++t) P += probs[(size_t)t * E + e];
        P /= (double)T;
        double f = (double)counts[e] / ((double)T * (double)k);
        aux += f * P;
    }
    return (double)E * aux;
}

/* ------------------------------------------------------------------------ */
/* Activations.  GELU(tanh) and GELU(erf) after Hendrycks & Gimpel; ReLU;
 * silu(z) = z / (1 + e^-z). */
static double act_fn(int act, double z)
{
    switch (act) {
    case ORC_RELU: return z > 0.0 ? z : 0.0;
    case ORC_GELU_TANH: {
        const double c = sqrt(2.0 / M_PI);
        return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
    }
    case ORC_GELU_ERF: return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
    default: return z / (1.0 + exp(-z)); /* silu */
    }
}

double orc_act(int act, double z) { return act_fn(act, z); }

/* Step 7 -- one expert on one token.  Expert e is a two-layer MLP ([Intro]
 * §3.2: Linear -> GELU -> Linear; [Sparse] §3.1), weights in nn.Linear
 * layout: W1[e] is [F, d], W2[e] is [d, F].  SwiGLU uses W3[e] ([F, d]) as
 * the linear branch.  xr is the token's row (d doubles), h scratch of F,
 * out receives d doubles. */
static void expert_ffn(int d, int F, int act, int e,
                       const void* W1, const void* W3, const void* W2, int wc,
                       const void* b1, const void* b2, int bc,
                       const double* xr, double* h, double* out)
{
    const size_t w1 = (size_t)e * F * d;
    for (int f = 0; f < F; ++f) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += rd(W1, wc, w1 + (size_t)f * d + i) * xr[i];
        if (b1) a += rd(b1, bc, (size_t)e * F + f);
        if (act == ORC_SWIGLU) {
            double b = 0.0;
            for (int i = 0; i < d; ++i) b += rd(W3, wc, w1 + (size_t)f * d + i) * xr[i];
            h[f] = act_fn(ORC_SWIGLU, a) * b;
        } else {
            h[f] = act_fn(act, a);
        }
    }
    const size_t w2 = (size_t)e * d * F;
    for (int o = 0; o < d; ++o) {
        double s = 0.0;
        for (int f = 0; f < F; ++f) s += rd(W2, wc, w2 + (size_t)o * F + f) * h[f];
        if (b2) s += rd(b2, bc, (size_t)e * d + o);
        out[o] = s;
    }
}

/* Steps 7-9 -- layer output for a list of tokens.
 *   y[t] = sum over kept slots j of gates[t,j] * FFN_{idx[t,j]}(x[t])    ([Intro] §3.4, [Basic] third formula)
 *        + sum over shared experts s < S of FFN_{E+s}(x[t])               ([Switch] §"共享专家隔离": always on, gate 1)
 *        + pass(t) * x[t]                                                 ([Switch] §"专家容量": 0 + x = x)
 * pass(t) = 1 if residual_mode == 1; with residual_mode == 0 it is 1 only when
 * k >= 1 and every routed slot of t was dropped.  Expert arrays hold E + S
 * experts, routed first.  tokens lists n_rows token ids; y is [n_rows, d]. */
void orc_output_rows(int T, int d, int F, int E, int S, int k, int act, int residual_mode,
                     const void* x, int x_code,
                     const void* W1, const void* W3, const void* W2, int w_code,
                     const void* b1, const void* b2, int b_code,
                     const int32_t* idx, const double* gates, const uint8_t* dropped,
                     int n_rows, const int32_t* tokens, double* y)
{
    (void)T;
    (void)E;
    #pragma omp parallel
    {
        double* xr = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)F);
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        #pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n_rows; ++r) {
            const long t = tokens[r];
            double* yr = y + (size_t)r * d;
            for (int i = 0; i < d; ++i) {
                xr[i] = rd(x, x_code, (size_t)t * d + i);
                yr[i] = 0.0;
            }
            int n_dropped = 0;
            for (int j = 0; j < k; ++j) {
                size_t s = (size_t)t * k + j;
                if (dropped[s]) {
                    ++n_dropped;
                    continue;
                }
                expert_ffn(d, F, act, idx[s], W1, W3, W2, w_code, b1, b2, b_code, xr, h, o);
                for (int i = 0; i < d; ++i) yr[i] += gates[s] * o[i];
            }
            for (int sh = 0; sh < S; ++sh) {
                expert_ffn(d, F, act, E + sh, W1, W3, W2, w_code, b1, b2, b_code, xr, h, o);
                for (int i = 0; i < d; ++i) yr[i] += o[i];
            }
            int pass = residual_mode == 1 || (k >= 1 && n_dropped == k);
            if (pass)
                for (int i = 0; i < d; ++i) yr[i] += xr[i];
        }
        free(xr);
        free(h);
        free(o);
    }
}

/* Number of threads the parallel loops above use (reported with timings). */
int orc_num_threads(void)
{
    int n = 1;
    #pragma omp parallel
    {
        #pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

/* ======================================================================== */
/* Backward pass (training).  [Intro] §3.4-§3.5 trains the layer end to end:
 * total_loss = task_loss + coef * aux_loss, then total_loss.backward().
 * [Switch] §"负载均衡损失函数": in N * sum_i f_i P_i only P_i (the mean router
 * probability) is differentiable; f_i counts an argmax and is not.  The
 * discrete decisions (the top-k choice, capacity drops, pass-through) are
 * held fixed: gradients reach the router only through the gate values and
 * P_i, as automatic differentiation of the listings' forward would give.
 *
 * Given dy = dL/dy [T,d] and d_aux = dL/d aux, this returns dL/d of every
 * input: x, W_gate, b_gate, W1, W3, W2, b1, b2 and, under noisy gating,
 * W_noise and b_noise (the normal draws are data, not parameters).  The
 * forward quantities are recomputed here in double precision from the
 * inputs; idx and dropped are the forward's decisions. */

/* d act / dz, from the definitions of act_fn (silu for SwiGLU). */
static double act_grad(int act, double z)
{
    switch (act) {
    case ORC_RELU: return z > 0.0 ? 1.0 : 0.0; /* the subgradient 0 at z = 0 */
    case ORC_GELU_TANH: {
        const double c = sqrt(2.0 / M_PI), a = 0.044715;
        const double th = tanh(c * (z + a * z * z * z));
        return 0.5 * (1.0 + th) + 0.5 * z * (1.0 - th * th) * c * (1.0 + 3.0 * a * z * z);
    }
    case ORC_GELU_ERF:
        return 0.5 * (1.0 + erf(z / sqrt(2.0))) + z * exp(-0.5 * z * z) / sqrt(2.0 * M_PI);
    default: {
        const double s = 1.0 / (1.0 + exp(-z));
        return s * (1.0 + z * (1.0 - s));
    }
    }
}

double orc_act_grad(int act, double z) { return act_grad(act, z); }

/* Router quantities of token t in double: clean logits l, noise logits n and
 * the logits the gating used (lg = l, or l + eps * (softplus(n) + min_std)). */
static void router_row(int d, int E, long t, const void* x, int xc, const void* wg, int wgc,
                       const void* bg, int bgc, const void* wn, const void* bn, const void* eps,
                       int nc, double min_std, double* l, double* n, double* lg)
{
    for (int e = 0; e < E; ++e) {
        double s = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
            const double xv = rd(x, xc, (size_t)t * d + i);
            s += xv * rd(wg, wgc, (size_t)e * d + i);
            if (wn) u += xv * rd(wn, nc, (size_t)e * d + i);
        }
        if (bg) s += rd(bg, bgc, (size_t)e);
        if (wn && bn) u += rd(bn, nc, (size_t)e);
        l[e] = s;
        n[e] = u;
        lg[e] = wn ? s + rd(eps, nc, (size_t)t * E + e) * (orc_softplus(u) + min_std) : s;
    }
}

void orc_backward(int T, int d, int F, int E, int S, int k, int act, int renormalize, int residual_mode,
                  const void* x, int x_code, const void* wg, int wg_code, const void* bg, int bg_code,
                  const void* W1, const void* W3, const void* W2, int w_code,
                  const void* b1, const void* b2, int b_code,
                  const void* wn, const void* bn, const void* eps, int n_code, double min_std,
                  const int32_t* idx, const uint8_t* dropped, const double* dy, double d_aux,
                  double* dx, double* dwg, double* dbg, double* dw1, double* dw3, double* dw2,
                  double* db1, double* db2, double* dwn, double* dbn)
{
    const int ES = E + S;
    const size_t slots = (size_t)T * k;
    /* gradient reaching each routed slot's gate, and each slot's input gradient */
    double* dg = (double*)calloc(slots, sizeof(double));
    double* dx_slot = (double*)calloc((slots + (size_t)T * S) * d, sizeof(double));
    double* gate = (double*)malloc(sizeof(double) * slots);
    double* probs = (double*)malloc(sizeof(double) * (size_t)T * E);
    double* nlog = (double*)malloc(sizeof(double) * (size_t)T * E);
    double* dl = (double*)calloc((size_t)T * E, sizeof(double));
    double* dn = (double*)calloc((size_t)T * E, sizeof(double));
    long long* counts = (long long*)calloc((size_t)E, sizeof(long long));

    /* forward router: probabilities and gates ([Basic] softmax, [Intro] §3.3 gates) */
    #pragma omp parallel
    {
        double* l = (double*)malloc(sizeof(double) * (size_t)E);
        double* lg = (double*)malloc(sizeof(double) * (size_t)E);
        #pragma omp for schedule(static)
        for (long t = 0; t < T; ++t) {
            router_row(d, E, t, x, x_code, wg, wg_code, bg, bg_code, wn, bn, eps, n_code, min_std, l,
                       nlog + (size_t)t * E, lg);
            double m = lg[0], den = 0.0;
            for (int e = 1; e < E; ++e)
                if (lg[e] > m) m = lg[e];
            for (int e = 0; e < E; ++e) den += exp(lg[e] - m);
            double* p = probs + (size_t)t * E;
            for (int e = 0; e < E; ++e) p[e] = exp(lg[e] - m) / den;
            double sel = 0.0;
            for (int j = 0; j < k; ++j) sel += p[idx[(size_t)t * k + j]];
            for (int j = 0; j < k; ++j) {
                const double pj = p[idx[(size_t)t * k + j]];
                gate[(size_t)t * k + j] = renormalize ? pj / sel : pj;
            }
        }
        free(l);
        free(lg);
    }
    for (size_t s = 0; s < slots; ++s) counts[idx[s]]++;

    /* experts, one at a time in parallel: every weight gradient of expert e is
     * private to its iteration.  do = gate * dy (gate 1 for shared experts). */
    memset(dw1, 0, sizeof(double) * (size_t)ES * F * d);
    if (dw3) memset(dw3, 0, sizeof(double) * (size_t)ES * F * d);
    memset(dw2, 0, sizeof(double) * (size_t)ES * d * F);
    if (db1) memset(db1, 0, sizeof(double) * (size_t)ES * F);
    if (db2) memset(db2, 0, sizeof(double) * (size_t)ES * d);
    #pragma omp parallel
    {
        double* xr = (double*)malloc(sizeof(double) * (size_t)d);
        double* z1 = (double*)malloc(sizeof(double) * (size_t)F);
        double* z3 = (double*)malloc(sizeof(double) * (size_t)F);
        double* h = (double*)malloc(sizeof(double) * (size_t)F);
        double* dh = (double*)malloc(sizeof(double) * (size_t)F);
        double* dz1 = (double*)malloc(sizeof(double) * (size_t)F);
        double* dz3 = (double*)malloc(sizeof(double) * (size_t)F);
        double* dout = (double*)malloc(sizeof(double) * (size_t)d);
        #pragma omp for schedule(dynamic, 1)
        for (long e = 0; e < ES; ++e) {
            const int shared = e >= E;
            const size_t w1o = (size_t)e * F * d, w2o = (size_t)e * d * F;
            for (size_t s = 0; s < (shared ? (size_t)T : slots); ++s) {
                const long t = shared ? (long)s : (long)(s / k);
                if (!shared && (idx[s] != e || dropped[s])) continue;
                for (int i = 0; i < d; ++i) xr[i] = rd(x, x_code, (size_t)t * d + i);
                /* forward of the expert on this token */
                for (int f = 0; f < F; ++f) {
                    double a = 0.0, b = 0.0;
                    for (int i = 0; i < d; ++i) {
                        a += rd(W1, w_code, w1o + (size_t)f * d + i) * xr[i];
                        if (act == ORC_SWIGLU) b += rd(W3, w_code, w1o + (size_t)f * d + i) * xr[i];
                    }
                    if (b1) a += rd(b1, b_code, (size_t)e * F + f);
                    z1[f] = a;
                    z3[f] = b;
                    h[f] = act == ORC_SWIGLU ? act_fn(ORC_SWIGLU, a) * b : act_fn(act, a);
                }
                const double g = shared ? 1.0 : gate[s];
                const double* dyr = dy + (size_t)t * d;
                if (!shared) {
                    /* dL/dgate = <dy, expert output> */
                    double acc = 0.0;
                    for (int o = 0; o < d; ++o) {
                        double out = 0.0;
                        for (int f = 0; f < F; ++f) out += rd(W2, w_code, w2o + (size_t)o * F + f) * h[f];
                        if (b2) out += rd(b2, b_code, (size_t)e * d + o);
                        acc += dyr[o] * out;
                    }
                    dg[s] = acc;
                }
                for (int o = 0; o < d; ++o) dout[o] = g * dyr[o];
                /* second layer: out = W2 h + b2 */
                for (int f = 0; f < F; ++f) {
                    double a = 0.0;
                    for (int o = 0; o < d; ++o) a += rd(W2, w_code, w2o + (size_t)o * F + f) * dout[o];
                    dh[f] = a;
                }
                for (int o = 0; o < d; ++o) {
                    for (int f = 0; f < F; ++f) dw2[w2o + (size_t)o * F + f] += dout[o] * h[f];
                    if (db2) db2[(size_t)e * d + o] += dout[o];
                }
                /* activation */
                for (int f = 0; f < F; ++f) {
                    if (act == ORC_SWIGLU) {
                        dz1[f] = dh[f] * z3[f] * act_grad(ORC_SWIGLU, z1[f]);
                        dz3[f] = dh[f] * act_fn(ORC_SWIGLU, z1[f]);
                    } else {
                        dz1[f] = dh[f] * act_grad(act, z1[f]);
                        dz3[f] = 0.0;
                    }
                }
                /* first layer: z1 = W1 x + b1, z3 = W3 x */
                double* dxs = dx_slot + (shared ? slots + (size_t)t * S + (size_t)(e - E) : s) * d;
                for (int f = 0; f < F; ++f) {
                    if (db1) db1[(size_t)e * F + f] += dz1[f];
                    for (int i = 0; i < d; ++i) {
                        dw1[w1o + (size_t)f * d + i] += dz1[f] * xr[i];
                        if (act == ORC_SWIGLU) dw3[w1o + (size_t)f * d + i] += dz3[f] * xr[i];
                    }
                }
                for (int i = 0; i < d; ++i) {
                    double a = 0.0;
                    for (int f = 0; f < F; ++f) {
                        a += rd(W1, w_code, w1o + (size_t)f * d + i) * dz1[f];
                        if (act == ORC_SWIGLU) a += rd(W3, w_code, w1o + (size_t)f * d + i) * dz3[f];
                    }
                    dxs[i] = a;
                }
            }
        }
        free(xr);
        free(z1);
        free(z3);
        free(h);
        free(dh);
        free(dz1);
        free(dz3);
        free(dout);
    }

    /* router: gates -> probabilities -> logits (softmax Jacobian), plus the balance
     * statistic's P_e term: d aux / d p[t,e] = E * f_e / T with f_e = counts_e / (T k) */
    #pragma omp parallel
    {
        double* dp = (double*)malloc(sizeof(double) * (size_t)E);
        #pragma omp for schedule(static)
        for (long t = 0; t < T; ++t) {
            const double* p = probs + (size_t)t * E;
            for (int e = 0; e < E; ++e)
                dp[e] = d_aux * (double)E * ((double)counts[e] / ((double)T * k)) / (double)T;
            double sel = 0.0, dot = 0.0;
            for (int j = 0; j < k; ++j) {
                const size_t s = (size_t)t * k + j;
                sel += p[idx[s]];
                dot += dg[s] * p[idx[s]];
            }
            for (int j = 0; j < k; ++j) {
                const size_t s = (size_t)t * k + j;
                /* renormalised: g_j = p_j / sum_sel p, so dp_i = dg_i / sel - sum_j dg_j p_j / sel^2 */
                dp[idx[s]] += renormalize ? dg[s] / sel - dot / (sel * sel) : dg[s];
            }
            double pdp = 0.0;
            for (int e = 0; e < E; ++e) pdp += p[e] * dp[e];
            for (int e = 0; e < E; ++e) {
                const double g = p[e] * (dp[e] - pdp);
                dl[(size_t)t * E + e] = g;
                if (wn) {
                    /* d/dn of eps * softplus(n) is eps * sigmoid(n) */
                    const double u = nlog[(size_t)t * E + e];
                    dn[(size_t)t * E + e] = g * rd(eps, n_code, (size_t)t * E + e) / (1.0 + exp(-u));
                }
            }
        }
        free(dp);
    }

    /* dx: expert slots + shared experts + pass-through + router (+ noise projection) */
    #pragma omp parallel for schedule(static)
    for (long t = 0; t < T; ++t) {
        int n_dropped = 0;
        for (int j = 0; j < k; ++j) n_dropped += dropped[(size_t)t * k + j] ? 1 : 0;
        const int pass = residual_mode == 1 || (k >= 1 && n_dropped == k);
        for (int i = 0; i < d; ++i) {
            double a = pass ? dy[(size_t)t * d + i] : 0.0;
            for (int j = 0; j < k; ++j) {
                const size_t s = (size_t)t * k + j;
                if (!dropped[s]) a += dx_slot[s * d + i];
            }
            for (int sh = 0; sh < S; ++sh) a += dx_slot[(slots + (size_t)t * S + sh) * d + i];
            for (int e = 0; e < E; ++e) {
                a += dl[(size_t)t * E + e] * rd(wg, wg_code, (size_t)e * d + i);
                if (wn) a += dn[(size_t)t * E + e] * rd(wn, n_code, (size_t)e * d + i);
            }
            dx[(size_t)t * d + i] = a;
        }
    }

    /* router weights: dW[e,i] = sum_t dl[t,e] x[t,i], db[e] = sum_t dl[t,e] */
    #pragma omp parallel for schedule(static)
    for (long e = 0; e < E; ++e) {
        for (int i = 0; i < d; ++i) {
            double a = 0.0, u = 0.0;
            for (long t = 0; t < T; ++t) {
                const double xv = rd(x, x_code, (size_t)t * d + i);
                a += dl[(size_t)t * E + e] * xv;
                u += dn[(size_t)t * E + e] * xv;
            }
            dwg[(size_t)e * d + i] = a;
            if (dwn) dwn[(size_t)e * d + i] = u;
        }
        double a = 0.0, u = 0.0;
        for (long t = 0; t < T; ++t) {
            a += dl[(size_t)t * E + e];
            u += dn[(size_t)t * E + e];
        }
        if (dbg) dbg[e] = a;
        if (dbn) dbn[e] = u;
    }

    free(dg);
    free(dx_slot);
    free(gate);
    free(probs);
    free(nlog);
    free(dl);
    free(dn);
    free(counts);
}

/* ======================================================================== */
/* Expert weight quantisation to int8.  [Arch] §"部署实践" converts expert
 * weights to 8-bit integers with almost no loss of accuracy; [Sparse]
 * §"量化与PagedAttention结合" quantises the experts while the router keeps its
 * precision.  The pages give no scheme; the plainest reading is symmetric
 * per-output-row quantisation with a real scale:
 *     scale[r] = max_c |w[r,c]| / 127,   q[r,c] = round(w[r,c] / scale[r])
 * (round half to even, |q| <= 127; an all-zero row gets scale 0 and q 0), and
 * the dequantised weight is q * scale.  The integer is decided by floating
 * point, so this function takes that decision in the precision the library
 * uses, IEEE fp32 (correctly rounded division, then rint), as the test rules
 * for integer results require; everything else here is plain. */
void orc_quantize_int8(int rows, int cols, const void* w, int w_code, int8_t* q, float* scale)
{
    for (long r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            const float v = (float)rd(w, w_code, (size_t)r * cols + c);
            const float a = v < 0.0f ? -v : v;
            if (a > amax) amax = a;
        }
        const float s = amax / 127.0f;
        scale[r] = s;
        for (int c = 0; c < cols; ++c) {
            const float v = (float)rd(w, w_code, (size_t)r * cols + c);
            float t = s > 0.0f ? rintf(v / s) : 0.0f;
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            q[(size_t)r * cols + c] = (int8_t)t;
        }
    }
}

/* ======================================================================== */
/* Expert parallelism over G ranks.  [Arch] §3.2 "分布式训练优化": experts are
 * placed on different devices; in the mixed data + expert parallel mode the
 * data is sharded over the workers, every worker holds a part of the experts,
 * and tokens are sent between devices.  [Sparse] §4.2 "专家分片": 64 experts
 * cut over 4 cards, 16 on each.  [Arch] §5 (问题3) names the exchange: an
 * AllToAll.  [Intro] §4 (第四): every token may be sent to another device.
 *
 * Readings (the pages give no layout):
 *   - rank r holds the tokens [floor(r T / G), floor((r+1) T / G)) and the
 *     experts [r E/G, (r+1) E/G); E is a multiple of G;
 *   - routing is per token, so a rank routes its own tokens exactly as the
 *     whole layer would;
 *   - capacity is the pages' rule applied to each shard on its own:
 *     C_r = floor(T_r cf / E), positions counted in the shard's token order;
 *   - every kept slot is sent to the rank that owns its expert; a rank's
 *     receive buffer holds its experts in ascending order and, inside one
 *     expert, the rows sent by rank 0, 1, ..., each in token order;
 *   - the expert outputs return to the token's rank, which combines them;
 *     shared experts are applied by each rank to its own tokens;
 *   - the balance statistic is reduced over all ranks: f_e and P_e are sums
 *     over every rank's tokens divided by T k and T. */

/* The exchange.  idx [T,k]; C_rank [G] (-1 = no limit).  Writes
 *   counts_rank [G,E]  slots of rank r's tokens that chose e (before drops)
 *   dropped [T,k]      per-shard capacity drops
 *   recv_row [T,k]     row of the slot in the concatenated receive buffers
 *                      (rank 0's rows first), -1 if dropped
 *   recv_rows [G]      rows each rank receives
 *   recv_slot [...]    for each row of the concatenated receive buffers, the
 *                      slot t*k + j it holds (sum of recv_rows entries). */
void orc_ep_exchange(int T, int E, int k, int G, const int32_t* idx, const long long* C_rank,
                     int32_t* counts_rank, uint8_t* dropped, int32_t* recv_row, int32_t* recv_rows,
                     int32_t* recv_slot)
{
    long long* seen = (long long*)calloc((size_t)E, sizeof(long long));
    const int E_loc = E / G;
    for (int r = 0; r < G; ++r) {
        const long t0 = (long)((long long)r * T / G), t1 = (long)((long long)(r + 1) * T / G);
        for (int e = 0; e < E; ++e) {
            seen[e] = 0;
            counts_rank[(size_t)r * E + e] = 0;
        }
        for (long t = t0; t < t1; ++t) {
            for (int j = 0; j < k; ++j) {
                const size_t s = (size_t)t * k + j;
                const int e = idx[s];
                counts_rank[(size_t)r * E + e] += 1;
                const long long p = seen[e]++;
                dropped[s] = (uint8_t)(C_rank[r] >= 0 && p >= C_rank[r]);
                recv_row[s] = -1;
            }
        }
    }
    long long row = 0;
    for (int q = 0; q < G; ++q) {
        long long n_q = 0;
        for (int e = q * E_loc; e < (q + 1) * E_loc; ++e) {
            for (int src = 0; src < G; ++src) {
                const long t0 = (long)((long long)src * T / G), t1 = (long)((long long)(src + 1) * T / G);
                for (long t = t0; t < t1; ++t) {
                    for (int j = 0; j < k; ++j) {
                        const size_t s = (size_t)t * k + j;
                        if (idx[s] != e || dropped[s]) continue;
                        recv_row[s] = (int32_t)row;
                        recv_slot[row] = (int32_t)s;
                        ++row;
                        ++n_q;
                    }
                }
            }
        }
        recv_rows[q] = (int32_t)n_q;
    }
    free(seen);
}

/* The owners' expert computation on a list of rows: out[r] = FFN_{expert[r]}(x[token[r]])
 * ([Intro] §3.2 two-layer MLP; shared experts are experts E..E+S-1).  out is
 * [n_rows, d]. */
void orc_expert_apply(int d, int F, int act, const void* x, int x_code,
                      const void* W1, const void* W3, const void* W2, int w_code,
                      const void* b1, const void* b2, int b_code,
                      int n_rows, const int32_t* token, const int32_t* expert, double* out)
{
    #pragma omp parallel
    {
        double* xr = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)F);
        #pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n_rows; ++r) {
            for (int i = 0; i < d; ++i) xr[i] = rd(x, x_code, (size_t)token[r] * d + i);
            expert_ffn(d, F, act, expert[r], W1, W3, W2, w_code, b1, b2, b_code, xr, h,
                       out + (size_t)r * d);
        }
        free(xr);
        free(h);
    }
}

/* The combine at the token's own rank after the return exchange, for the
 * tokens listed in `tokens` (y is [n_tok, d]):
 *   y[t] = sum over kept slots j (slot order) of gates[t,j] * o[row_of[t,j]]
 *        + sum over shared experts s of ys[s, t] + pass(t) x[t]
 * with row_of[t,j] the slot's row in o (the concatenated receive buffers'
 * outputs), ys [S, T, d] the shared experts' outputs (may be NULL when S = 0),
 * and pass(t) as in orc_output_rows. */
void orc_ep_combine(int T, int d, int k, int S, int residual_mode, const void* x, int x_code,
                    const double* gates, const uint8_t* dropped, const int32_t* row_of, const double* o,
                    const double* ys, int n_tok, const int32_t* tokens, double* y)
{
    for (long r = 0; r < n_tok; ++r) {
        const long t = tokens[r];
        double* yr = y + (size_t)r * d;
        for (int i = 0; i < d; ++i) yr[i] = 0.0;
        int n_dropped = 0;
        for (int j = 0; j < k; ++j) {
            const size_t s = (size_t)t * k + j;
            if (dropped[s]) {
                ++n_dropped;
                continue;
            }
            const double* orow = o + (size_t)row_of[s] * d;
            for (int i = 0; i < d; ++i) yr[i] += gates[s] * orow[i];
        }
        for (int sh = 0; sh < S; ++sh)
            for (int i = 0; i < d; ++i) yr[i] += ys[((size_t)sh * T + t) * d + i];
        if (residual_mode == 1 || (k >= 1 && n_dropped == k))
            for (int i = 0; i < d; ++i) yr[i] += rd(x, x_code, (size_t)t * d + i);
    }
}

/* The balance statistic reduced over the ranks (an all-reduce of each rank's
 * counts and probability sums): E * sum_e f_e P_e with
 * f_e = (sum_r counts_rank[r,e]) / (T k) and P_e = (sum_r sum_{t in shard r} p[t,e]) / T
 * ([Intro] §3.4, [Switch] §"负载均衡损失函数"). */
double orc_ep_aux(int T, int E, int k, int G, const int32_t* counts_rank, const double* probs)
{
    double aux = 0.0;
    for (int e = 0; e < E; ++e) {
        long long c = 0;
        double P = 0.0;
        for (int r = 0; r < G; ++r) {
            c += counts_rank[(size_t)r * E + e];
            const long t0 = (long)((long long)r * T / G), t1 = (long)((long long)(r + 1) * T / G);
            double Pr = 0.0;
            for (long t = t0; t < t1; ++t) Pr += probs[(size_t)t * E + e];
            P += Pr;
        }
        aux += ((double)c / ((double)T * (double)k)) * (P / (double)T);
    }
    return (double)E * aux;
}

/* ======================================================================== */
/* Expert weight quantisation to 4 bits.  [Sparse] §"量化与PagedAttention结合":
 * the expert weights may be quantised on their own (for example to INT4, with
 * AWQ) while the router keeps 16-bit precision.  The pages give no scheme.
 * AWQ stores 4-bit weights in groups of consecutive input elements, each
 * group with its own scale; its activation-aware choice of the scales needs
 * calibration data, which this layer does not have, so the reading here is
 * the plain group-wise rounding that remains:
 *     scale[r, g] = max over the group's elements |w[r, c]| / 7,
 *     q[r, c] = round(w[r, c] / scale[r, g]) clamped to [-7, 7]
 * for groups of `group` consecutive columns c (round half to even; an
 * all-zero group gets scale 0 and q 0); the dequantised weight is
 * q * scale.  As for int8, the integer is decided in IEEE fp32 (the
 * library's precision).  Two values share one byte: column 2i in the low
 * nibble, 2i + 1 in the high nibble, each as a 4-bit two's complement. */
void orc_quantize_int4(int rows, int cols, int group, const void* w, int w_code, uint8_t* packed, float* scale)
{
    const int n_groups = cols / group;
    for (long r = 0; r < rows; ++r) {
        for (int g = 0; g < n_groups; ++g) {
            float amax = 0.0f;
            for (int c = g * group; c < (g + 1) * group; ++c) {
                const float v = (float)rd(w, w_code, (size_t)r * cols + c);
                const float a = v < 0.0f ? -v : v;
                if (a > amax) amax = a;
            }
            const float s = amax / 7.0f;
            scale[(size_t)r * n_groups + g] = s;
            for (int c = g * group; c < (g + 1) * group; ++c) {
                const float v = (float)rd(w, w_code, (size_t)r * cols + c);
                float t = s > 0.0f ? rintf(v / s) : 0.0f;
                if (t > 7.0f) t = 7.0f;
                if (t < -7.0f) t = -7.0f;
                const uint8_t nib = (uint8_t)((int)t & 0xF);
                uint8_t* b = packed + (size_t)r * (cols / 2) + c / 2;
                if (c % 2 == 0) *b = (uint8_t)((*b & 0xF0u) | nib);
                else *b = (uint8_t)((*b & 0x0Fu) | (uint8_t)(nib << 4));
            }
        }
    }
}
