// grouped_gemm_wq.cu -- stage 3 with quantised expert weights (8-bit per-row or
// 4-bit group-wise) for layers whose experts see few tokens each, where the
// expert stage streams the weights from HBM.
//
// "MoE架构解析" §"部署实践": expert weights stored as 8-bit integers lose almost
// no accuracy and shrink the bytes the expert stage streams; "MoE混合专家模型
// 原理与实战" §"量化与PagedAttention结合": the experts alone may be quantised to
// INT4 (AWQ: group-wise scales) while the router keeps its precision.
//
// The kernel computes the transposed product, with the weights as the MMA's A
// operand taken from tensor memory:
//     D[n, m] = sum_k W[n, k] X[m, k]      (n: 128 weight rows, m: NT tokens)
// The converter warps read each landed weight tile from shared memory once,
// turn it into bf16 in registers and write it straight into TMEM
// (tcgen05.st), so the converted operand never makes a round trip through
// shared memory; the tensor core reads A from TMEM and the token tile (B,
// K-major, 128-byte swizzle) from shared memory.  The token tile is small
// (NT = 32 .. 128 rows, as many as the experts hold), so no MMA work is spent
// on padding rows of 128-row token tiles.  Each weight is converted once per
// token tile, so NT covers all the rows an expert holds where it can.
//   8-bit: q in [-127, 127] is exact in bf16; the per-row scale is applied to
//          the accumulator in the epilogue: sum_k q[n,k] x[m,k] * scale[n].
//   4-bit: the converter multiplies q in [-7, 7] by its group's scale (groups
//          of 128 input columns) in packed bf16 arithmetic: bf16(q * bf16(s)).
// Two A tiles share each token tile: with SwiGLU the W1 and W3 tiles of the same
// 128 rows (the epilogue pairs their accumulators), otherwise (NT <= 96, PAIR) two
// consecutive 128-row tiles, so a tile covers 256 weight rows.  One thread of the
// epilogue holds one weight row (its TMEM lane) of each A tile for NT tokens:
// scale, bias and activation are per-thread scalars.
//
// Per CTA (one per SM, 512 threads):
//   warp 0      TMA, per shared-memory stage of KS = 128 (8-bit) or 256 (4-bit) K
//               values: the weight tile(s) [128 rows x 128 bytes] (128-byte swizzle:
//               every row segment a copy fetches is 128 contiguous bytes of HBM) and
//               the token tile as KS / 64 boxes [NT x 64] bf16;
//   warp 1      TMEM allocation and tcgen05.mma (M = 128, N = NT, K = 16, A from TMEM);
//   warps 4-11  converters, two per TMEM lane quarter (warp w writes lanes
//               32 (w % 4) .. + 31): with two A tiles each converts one of them,
//               otherwise each converts one half of the K block; one TMEM store
//               stays in flight while the next sub-block is converted;
//   warps 12-15 epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31).
// The shared-memory stages (S, as many as fit: they keep the weight stream's bytes
// in flight) and the TMEM operand slots (NA of 64 K values each, as many as the
// accumulators leave) are separate rings: a stage feeds KS / 64 slots; it is refilled
// once the MMAs that read its token tile are done, a slot is rewritten once the MMAs
// that read it are done.
// Every wait is bounded, as in the other tcgen05 kernels.
#include "common.cuh"
#include "kernels.h"
#include "tc_tile.cuh"

namespace moe {

namespace {

constexpr int kBW = 128;  // weight rows per A tile (MMA M)
constexpr int kBK = 64;   // reduction per TMEM operand slot
constexpr int kThreads = 512;
constexpr int kConvWarps = 8;
constexpr int kGroupCols = 128;  // 4-bit scale groups along K
constexpr size_t kBarBytes = 512;
constexpr size_t kTableBytes = sizeof(int) * (3 * kMaxExperts + 2);
constexpr size_t kSmemBudget = 200 * 1024;  // shared-memory stages

template <int WBITS, bool TWO, int NT>
struct Cfg {
    static_assert(NT % 32 == 0, "token tile");
    static constexpr int kNA = TWO ? 2 : 1;                      // A tiles per K block
    static constexpr int kKS = WBITS == 8 ? 128 : 256;           // K values per shared-memory stage
    static constexpr int kSub = kKS / kBK;                       // TMEM slots per stage
    static constexpr uint32_t kXBoxBytes = NT * kBK * 2;         // one [NT x 64] token box
    static constexpr uint32_t kXBytes = kSub * kXBoxBytes;       // the stage's token tile
    static constexpr uint32_t kWRowBytes = kKS * WBITS / 8;      // 128 bytes
    static constexpr uint32_t kWBytes = kNA * kBW * kWRowBytes;  // weight tile(s)
    static constexpr uint32_t kStageBytes = (kXBytes + kWBytes + 1023) / 1024 * 1024;
    static constexpr int kStagesFit = (int)(kSmemBudget / kStageBytes);
    static constexpr int kStages = kStagesFit > 12 ? 12 : kStagesFit;  // shared-memory stages
    static constexpr uint32_t kAccCols = kNA * NT;               // one accumulator set
    static constexpr uint32_t kACols = kNA * 32;                 // TMEM A columns per slot
    static constexpr uint32_t kACol0 = 2 * kAccCols;             // A slots after the two accumulators
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kSlotsFit = (int)((kTmemCols - kACol0) / kACols);
    static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;  // TMEM operand slots
    static_assert(kSlots >= 2 && kStages >= 2, "pipeline depth");
    static_assert(2 * (kStages + kSlots) + 5 <= (int)(kBarBytes / 8) - 2, "barrier space");
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes + kTableBytes;
};

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Each thread of the warp stores 32 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Each thread of the warp stores 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// int8 x 4 (one 32-bit word) -> bf16 x 4 (two words), exactly, in packed bf16x2
// arithmetic: a two's-complement byte is v = m - 128 s (m its low seven bits, s its
// top bit).  With the high byte 0x43, m in the low byte is the bf16 128 + m (seven
// mantissa bits) and s moved to bit 7 is the bf16 128 or 256 (the exponent's lowest
// bit), so one packed subtraction leaves v, an integer of magnitude <= 128 (exact).
__device__ __forceinline__ void i8x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    const uint32_t wm = w & 0x7F7F7F7Fu;  // m of each byte
    const uint32_t ws = w & 0x80808080u;  // s of each byte, at bit 7
    // byte pairs (0, 1) and (2, 3), each byte below the constant 0x43
    const uint32_t a01 = __byte_perm(wm, 0x43u, 0x4140u), a23 = __byte_perm(wm, 0x43u, 0x4342u);
    const uint32_t b01 = __byte_perm(ws, 0x43u, 0x4140u), b23 = __byte_perm(ws, 0x43u, 0x4342u);
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(a01), "r"(b01));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(a23), "r"(b23));
}

// int4 x 8 (one 32-bit word; byte j holds value 2j in its low nibble, 2j + 1 in its
// high nibble) -> bf16 x 8 of q * s (four words), in packed bf16x2 arithmetic.  Offset
// binary n = q + 8 (flip each nibble's top bit).  Per byte j one byte permute puts byte j
// of u in the low half and byte j of u >> 1 in the high half, each below the constant
// 0x43 byte, and one mask keeps the low nibble (bits 0-3: bf16 128 + n_2j) and the
// shifted high nibble (bits 3-6: bf16 128 + 8 n_2j+1).  A packed subtraction of
// {136, 192} leaves {q_2j, 8 q_2j+1} exactly, and a packed multiply by
// s2 = {bf16(s), bf16(s) / 8} gives bf16(q * bf16(s)) in both halves (the division by 8
// is exact, so 8 q * (s / 8) = q * s before the one rounding).
__device__ __forceinline__ void i4x8_to_bf16(uint32_t w, uint32_t s2, uint32_t (&o)[4])
{
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t u1 = u >> 1;
    const uint32_t k_off = 0x43404308u;  // bf16 {low: 136, high: 192}
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        // byte 0 = u.p, byte 2 = u1.p (bytes 1 and 3 are cleared by the mask, which
        // also sets them to 0x43)
        const uint32_t v = __byte_perm(u, u1, (uint32_t)p | ((uint32_t)(4 + p) << 8));
        uint32_t m;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(m) : "r"(v), "r"(0x0078000Fu), "r"(0x43004300u));
        uint32_t q;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(m), "r"(k_off));
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[p]) : "r"(q), "r"(s2));
    }
}

// Tiles: group g has tt[g] = ceil(rows[g] / NT) token tiles and n_tiles weight-row
// tiles; inside a group the token tile runs fastest, so the CTAs working at the same
// time share each weight tile through L2.
struct WqTiles {
    int g = 0;
    __device__ __forceinline__ void locate(int tile, const int* toff, int n_tiles, int& mt, int& n)
    {
        while (tile >= toff[g + 1] * n_tiles) ++g;
        const int local = tile - toff[g] * n_tiles;
        const int ttg = toff[g + 1] - toff[g];
        n = local / ttg;
        mt = local - n * ttg;
    }
};

// PAIR (layers without SwiGLU): a tile is 256 weight rows, two A tiles of 128 rows
// against one token tile, so each token tile is loaded half as often and every
// converter warp turns a whole 64-value sub-block of one A tile into bf16 (as with
// SwiGLU's W1 / W3 pair).
template <int WBITS, int ACT, int NT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    k_grouped_gemm_wq(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmW3, const GroupedGemmWqArgs args)
{
    constexpr bool GATED = (ACT == kActSwiglu);
    static_assert(!(GATED && PAIR), "SwiGLU already pairs W1 and W3");
    constexpr bool TWO = GATED || PAIR;               // two A tiles per K block
    constexpr int kTileRows = PAIR ? 2 * kBW : kBW;   // weight rows per tile
    using C = Cfg<WBITS, TWO, NT>;
    constexpr int S = C::kStages;
    constexpr int NA = C::kSlots;
    constexpr uint32_t IDESC = idesc_bf16_f32(kBW, NT);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_q = reinterpret_cast<uint64_t*>(base + (size_t)S * C::kStageBytes);  // [S] stage landed
    uint64_t* empty = full_q + S;                                                      // [S] stage consumed
    uint64_t* full_a = empty + S;                                                      // [NA] slot written
    uint64_t* a_empty = full_a + NA;                                                   // [NA] slot consumed
    uint64_t* tfull = a_empty + NA;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_toff = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full_q) + kBarBytes);  // [G + 1]
    int* s_roff = s_toff + kMaxExperts + 1;
    int* s_rows = s_roff + kMaxExperts;

    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_q[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < NA; ++a) {
            mbar_init(&full_a[a], kConvWarps);  // one arrival per converter warp
            mbar_init(&a_empty[a], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (GATED) tma_prefetch_desc(&tmW3);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();  // segment tables and the token rows come from earlier kernels
    for (int i = threadIdx.x; i < G; i += kThreads) {
        s_roff[i] = args.row_off[i];
        s_rows[i] = args.rows[i];
    }
    __syncthreads();
    if (warp == 0) {  // token-tile offsets: exclusive prefix of ceil(rows / NT) over the groups
        const int per = (G + 31) / 32;
        const int b = lane * per, e = min(G, b + per);
        int sum = 0;
        for (int i = b; i < e; ++i) sum += (s_rows[i] + NT - 1) / NT;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int run = incl - sum;
        for (int i = b; i < e; ++i) {
            s_toff[i] = run;
            run += (s_rows[i] + NT - 1) / NT;
        }
        if (lane == 31) s_toff[G] = incl;
    }
    __syncthreads();

    const int n_tiles = args.n_tiles;
    const int total = s_toff[G] * n_tiles;
    const int num_kb = ceil_div(args.K, C::kKS);  // shared-memory stages per tile

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, filled = 0, fill_par = 0;
            bool ok = true;
            WqTiles tm;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int mt, n;
                tm.locate(tile, s_toff, n_tiles, mt, n);
                const int x_row = s_roff[tm.g] + mt * NT;
                const int w_row = tm.g * args.b_rows_per_group + n * kTileRows;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = base + (size_t)stage * C::kStageBytes;
                    mbar_arrive_expect_tx(&full_q[stage], C::kXBytes + C::kWBytes);
#pragma unroll
                    for (int u = 0; u < C::kSub; ++u)
                        tma_load_2d(st + u * C::kXBoxBytes, &tmX, &full_q[stage], kb * C::kKS + u * kBK, x_row,
                                    pol_act);
                    const int wc = kb * (int)C::kWRowBytes;  // byte column of the weight rows
                    tma_load_2d(st + C::kXBytes, &tmW, &full_q[stage], wc, w_row, pol_w);
                    if (GATED) tma_load_2d(st + C::kXBytes + kBW * C::kWRowBytes, &tmW3, &full_q[stage], wc, w_row, pol_w);
                    if (PAIR) tma_load_2d(st + C::kXBytes + kBW * C::kWRowBytes, &tmW, &full_q[stage], wc, w_row + kBW, pol_w);
                    filled |= 1u << stage;
                    fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutProducer);
                *abort_flag = 1;
                for (int s = 0; s < S; ++s)
                    if (((filled >> s) & 1u) && !mbar_wait_short(&full_q[s], (fill_par >> s) & 1u))
                        atomicOr(args.err, kErrTimeoutDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            int slot = 0;
            uint32_t sphase = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
                for (int kb = 0; kb < num_kb && ok; ++kb) {
                    const uint32_t xs = smem_u32(base + (size_t)stage * C::kStageBytes);
                    for (int u = 0; u < C::kSub; ++u) {
                        // the converters wrote this slot after the stage's TMA landed, so the
                        // token tile of the stage is in shared memory too
                        if (!mbar_wait(&full_a[slot], sphase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t x0 = xs + u * C::kXBoxBytes;
                        const uint32_t a0 = tmem_base + C::kACol0 + slot * C::kACols;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            const uint64_t bdesc = sdesc_kmajor_sw128(x0 + k * 32);
                            const uint32_t accum = (kb | u | k) != 0 ? 1u : 0u;
                            mma_bf16_ts(d_tmem, a0 + k * 8, bdesc, IDESC, accum);
                            if (TWO) mma_bf16_ts(d_tmem + NT, a0 + 32 + k * 8, bdesc, IDESC, accum);
                        }
                        mma_commit(&a_empty[slot]);
                        if (++slot == NA) {
                            slot = 0;
                            sphase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&tfull[acc]);
            }
            if (!ok) {
                atomicOr(args.err, kErrTimeoutMma);
                *abort_flag = 1;
            }
            mma_commit(drain);
            if (!mbar_wait_short(drain, 0)) atomicOr(args.err, kErrTimeoutDrain);
        }
    } else if (warp >= 4 && warp < 4 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int q = warp & 3;
        const int part = (warp - 4) >> 2;  // SwiGLU: the W1 / W3 tile; otherwise the K half
        const int r = q * 32 + lane;       // this thread's weight row in the tile (its TMEM lane)
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const int h = TWO ? part : 0;    // which weight tile of the stage
        const int kh = TWO ? -1 : part;  // which K half (-1: both)
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0;
        bool ok = true;
        // One TMEM store stays in flight while the next sub-block is converted: the
        // slot it wrote is signalled (wait::st, then the arrival) just before the next
        // store, and the last one after the loop.
        int pend = -1;
        WqTiles tm;
        const float* __restrict__ scales = (GATED && part == 1) ? args.scale3 : args.scale;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            int mt, n;
            tm.locate(tile, s_toff, n_tiles, mt, n);
            const int rr = n * kTileRows + (PAIR ? h * kBW : 0) + r;    // row within the group
            const int w_row = tm.g * args.b_rows_per_group + rr;         // global weight row
            const bool w_ok = rr < args.N;
            // 4-bit: the group scales of a stage's two 128-column groups, loaded one stage
            // ahead (each thread's scales are a separate sector, so the load is slow)
            const int ng = WBITS == 4 ? args.K / kGroupCols : 0;
            const float* srow = scales + (size_t)(w_ok ? w_row : 0) * ng;
            float nx0 = 0.0f, nx1 = 0.0f;
            if (WBITS == 4 && w_ok) {
                nx0 = __ldg(&srow[0]);
                if (1 < ng) nx1 = __ldg(&srow[1]);
            }
            for (int kb = 0; kb < num_kb && ok; ++kb) {
                const float sc0 = nx0, sc1 = nx1;
                if constexpr (WBITS == 4) {
                    const int g1 = ((kb + 1) * C::kKS) / kGroupCols;  // the next stage's first group
                    if (w_ok && g1 < ng) {
                        nx0 = __ldg(&srow[g1]);
                        if (g1 + 1 < ng) nx1 = __ldg(&srow[g1 + 1]);
                    }
                }
                if (!mbar_wait(&full_q[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                // this thread's 128-byte weight row; 16-byte chunk c sits at c ^ (r % 8)
                const uint8_t* row = base + (size_t)stage * C::kStageBytes + C::kXBytes +
                                     (size_t)(h * kBW + r) * C::kWRowBytes;
                for (int u = 0; u < C::kSub; ++u) {
                    uint32_t v[32];
                    // 16-byte chunks of sub-block u (64 K values) that this thread converts
                    constexpr int kChunks = WBITS == 8 ? 4 : 2;
                    const int cbase = u * kChunks + (kh < 0 ? 0 : kh * (kChunks / 2));
#pragma unroll
                    for (int ci = 0; ci < (TWO ? kChunks : kChunks / 2); ++ci) {
                        const int c = cbase + ci;
                        const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
                        if constexpr (WBITS == 8) {
                            i8x4_to_bf16(w.x, v[ci * 8 + 0], v[ci * 8 + 1]);
                            i8x4_to_bf16(w.y, v[ci * 8 + 2], v[ci * 8 + 3]);
                            i8x4_to_bf16(w.z, v[ci * 8 + 4], v[ci * 8 + 5]);
                            i8x4_to_bf16(w.w, v[ci * 8 + 6], v[ci * 8 + 7]);
                        } else {
                            const float scf = (u * kBK) / kGroupCols == 0 ? sc0 : sc1;
                            const float sb = __bfloat162float(__float2bfloat16_rn(scf));
                            const uint32_t scu = pack_bf16x2(sb, sb * 0.125f);  // {s, s / 8}, exact
                            uint32_t o[4];
                            i4x8_to_bf16(w.x, scu, o);
                            v[ci * 16 + 0] = o[0], v[ci * 16 + 1] = o[1], v[ci * 16 + 2] = o[2], v[ci * 16 + 3] = o[3];
                            i4x8_to_bf16(w.y, scu, o);
                            v[ci * 16 + 4] = o[0], v[ci * 16 + 5] = o[1], v[ci * 16 + 6] = o[2], v[ci * 16 + 7] = o[3];
                            i4x8_to_bf16(w.z, scu, o);
                            v[ci * 16 + 8] = o[0], v[ci * 16 + 9] = o[1], v[ci * 16 + 10] = o[2], v[ci * 16 + 11] = o[3];
                            i4x8_to_bf16(w.w, scu, o);
                            v[ci * 16 + 12] = o[0], v[ci * 16 + 13] = o[1], v[ci * 16 + 14] = o[2], v[ci * 16 + 15] = o[3];
                        }
                    }
                    if (pend >= 0) {  // the previous store has landed: its slot is ready for the MMA
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full_a[pend]);
                        pend = -1;
                    }
                    if (!mbar_wait(&a_empty[slot], sphase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = t_row + C::kACol0 + slot * C::kACols + h * 32;
                    if constexpr (TWO) {
                        tmem_st_32cols(dst, v);  // the whole sub-block of one tile's row
                    } else {
                        tmem_st_16cols(dst + kh * 16, v);  // one K half of the sub-block
                    }
                    pend = slot;
                    if (++slot == NA) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        tmem_st_wait();  // no store in flight past this point (also on the abort path)
        if (pend >= 0 && ok) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[pend]);
        }
        if (!ok) {
            if (lane == 0) atomicOr(args.err, kErrTimeoutProducer);
            *abort_flag = 1;
        }
    } else if (warp >= 4 + kConvWarps) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int r = q * 32 + lane;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
        const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(args.bias);
        bool ok = true;
        int it = 0;
        WqTiles tm;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            int mt, n;
            tm.locate(tile, s_toff, n_tiles, mt, n);
            const int acc = it & 1;
            if (!mbar_wait(&tfull[acc], (it >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            // this thread's output column (PAIR: and the one 128 columns on, from the
            // second accumulator)
            const int col = n * kTileRows + r;
            const bool col_ok = col < args.N;
            const bool col2_ok = PAIR && col + kBW < args.N;
            const size_t wr = (size_t)tm.g * args.b_rows_per_group + (col_ok ? col : 0);
            const size_t wr2 = (size_t)tm.g * args.b_rows_per_group + (col2_ok ? col + kBW : 0);
            // per-row factors: the 8-bit scales (the 4-bit ones were applied by the converters)
            float f1 = 1.0f, f3 = 1.0f, b = 0.0f, b2 = 0.0f;
            if constexpr (WBITS == 8) {
                f1 = args.scale[wr];
                if (GATED) f3 = args.scale3[wr];
                if (PAIR) f3 = args.scale[wr2];
            }
            if (!GATED && bias != nullptr) {
                b = __bfloat162float(bias[wr]);
                if (PAIR) b2 = __bfloat162float(bias[wr2]);
            }
            const int m0 = mt * NT;
            const int valid = min(NT, s_rows[tm.g] - m0);
            __nv_bfloat16* o = out + (size_t)(s_roff[tm.g] + m0) * args.ldo + col;
            const uint32_t t_lane = tmem_base + acc * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
            constexpr int CH = NT < 32 ? NT : 32;  // accumulator columns per load
#pragma unroll 1
            for (int c = 0; c < NT / CH; ++c) {
                uint32_t va[CH], vb[CH];
                if constexpr (CH == 32) {
                    tmem_ld_32cols(t_lane + c * CH, va);
                    if constexpr (TWO) tmem_ld_32cols(t_lane + NT + c * CH, vb);
                } else {
                    tmem_ld_16cols(t_lane + c * CH, va);
                    if constexpr (TWO) tmem_ld_16cols(t_lane + NT + c * CH, vb);
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int m = c * CH + j;
                    float z = __uint_as_float(va[j]) * f1;
                    float y;
                    if constexpr (GATED) {
                        y = activate_bf16out<kActSwiglu>(z) * (__uint_as_float(vb[j]) * f3);
                    } else {
                        y = activate_bf16out<ACT>(z + b);
                    }
                    if (col_ok && m < valid) o[(size_t)m * args.ldo] = __float2bfloat16_rn(y);
                    if constexpr (PAIR) {
                        const float y2 = activate_bf16out<ACT>(__uint_as_float(vb[j]) * f3 + b2);
                        if (col2_ok && m < valid) o[(size_t)m * args.ldo + kBW] = __float2bfloat16_rn(y2);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        if (!ok) {
            if (lane == 0) atomicOr(args.err, kErrTimeoutEpilogue);
            *abort_flag = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int WBITS, int ACT, int NT, bool PAIR>
cudaError_t launch_t(const CUtensorMap& x, const CUtensorMap& w, const CUtensorMap& w3, const GroupedGemmWqArgs& a,
                     int grid, cudaStream_t st, bool pdl)
{
    using C = Cfg<WBITS, ACT == kActSwiglu || PAIR, NT>;
    auto kern = k_grouped_gemm_wq<WBITS, ACT, NT, PAIR>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), C::kSmem, st, pdl, x, w, w3, a);
}

// Two A tiles (SwiGLU, or PAIR) hold two accumulators of NT columns, double-buffered,
// beside at least two operand slots in the 512 TMEM columns: NT <= 96.
template <int WBITS, int NT>
cudaError_t launch_nt(const CUtensorMap& x, const CUtensorMap& w, const CUtensorMap& w3, const GroupedGemmWqArgs& a,
                      int act, int grid, cudaStream_t st, bool pdl)
{
    constexpr bool P = NT <= 96;
    switch (act) {
    case kActNone: return launch_t<WBITS, kActNone, NT, P>(x, w, w3, a, grid, st, pdl);
    case kActRelu: return launch_t<WBITS, kActRelu, NT, P>(x, w, w3, a, grid, st, pdl);
    case kActGeluTanh: return launch_t<WBITS, kActGeluTanh, NT, P>(x, w, w3, a, grid, st, pdl);
    case kActGeluErf: return launch_t<WBITS, kActGeluErf, NT, P>(x, w, w3, a, grid, st, pdl);
    default:
        if constexpr (NT <= 64) return launch_t<WBITS, kActSwiglu, NT, false>(x, w, w3, a, grid, st, pdl);
        return cudaErrorInvalidValue;  // the gated layer's tensor-memory budget caps NT at 64
    }
}

// One warp per (row, group of 128 columns): scale = max|w| / 7, q = rint(w / scale)
// (IEEE fp32 division) clamped to [-7, 7], two values per byte (low nibble first).
template <typename T>
__global__ void __launch_bounds__(256) k_quantize_int4(const T* __restrict__ w, long long rows, int cols,
                                                       uint8_t* __restrict__ q, float* __restrict__ scale)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ng = cols / kGroupCols;
    const long long items = rows * ng;
    for (long long it = (long long)blockIdx.x * 8 + warp; it < items; it += (long long)gridDim.x * 8) {
        const long long row = it / ng;
        const int g = (int)(it - row * ng);
        const T* src = w + row * cols + g * kGroupCols + lane * 4;
        float v[4];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = to_f32(src[i]);
            amax = fmaxf(amax, fabsf(v[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax / 7.0f;
        if (lane == 0) scale[it] = s;
        uint32_t nib[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float t = s > 0.0f ? rintf(v[i] / s) : 0.0f;
            t = fminf(fmaxf(t, -7.0f), 7.0f);
            nib[i] = static_cast<uint32_t>(static_cast<int>(t)) & 0xFu;
        }
        const uint16_t packed = static_cast<uint16_t>(nib[0] | (nib[1] << 4) | (nib[2] << 8) | (nib[3] << 12));
        *reinterpret_cast<uint16_t*>(q + row * (cols / 2) + g * (kGroupCols / 2) + lane * 2) = packed;
    }
}

}  // namespace

int gemm_wq_weight_tiles(int N, int act, int nt)
{
    const bool pair = act != kActSwiglu && nt <= 96;
    return ceil_div(N, pair ? 2 * kBW : kBW);
}

int gemm_wq_tokens_tile(int rows_per_expert, bool gated)
{
    if (rows_per_expert <= 32) return 32;
    if (rows_per_expert <= 64 || gated) return 64;
    if (rows_per_expert <= 96) return 96;
    return 128;
}

cudaError_t launch_gemm_wq(const CUtensorMap& x, const CUtensorMap& w, const CUtensorMap& w3,
                           const GroupedGemmWqArgs& a, int wbits, int act, int nt, int grid, cudaStream_t st, bool pdl)
{
    if (wbits == 8) {
        if (nt == 32) return launch_nt<8, 32>(x, w, w3, a, act, grid, st, pdl);
        if (nt == 64) return launch_nt<8, 64>(x, w, w3, a, act, grid, st, pdl);
        if (nt == 96) return launch_nt<8, 96>(x, w, w3, a, act, grid, st, pdl);
        return launch_nt<8, 128>(x, w, w3, a, act, grid, st, pdl);
    }
    if (nt == 32) return launch_nt<4, 32>(x, w, w3, a, act, grid, st, pdl);
    if (nt == 64) return launch_nt<4, 64>(x, w, w3, a, act, grid, st, pdl);
    if (nt == 96) return launch_nt<4, 96>(x, w, w3, a, act, grid, st, pdl);
    return launch_nt<4, 128>(x, w, w3, a, act, grid, st, pdl);
}

cudaError_t launch_quantize_int4(const void* w, bool bf16, long long rows, int cols, uint8_t* q, float* scale,
                                 int sms, cudaStream_t st)
{
    const long long items = rows * (cols / kGroupCols);
    long long grid = (items + 7) / 8;
    if (grid > (long long)sms * 32) grid = (long long)sms * 32;
    if (grid < 1) grid = 1;
    if (bf16)
        return launch_kernel(k_quantize_int4<__nv_bfloat16>, dim3((int)grid), dim3(256), 0, st, false,
                             static_cast<const __nv_bfloat16*>(w), rows, cols, q, scale);
    return launch_kernel(k_quantize_int4<float>, dim3((int)grid), dim3(256), 0, st, false,
                         static_cast<const float*>(w), rows, cols, q, scale);
}

}  // namespace moe
