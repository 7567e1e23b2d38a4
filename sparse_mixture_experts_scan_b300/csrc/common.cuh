// common.cuh -- shared device helpers of the B300 MoE library (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor), and the
// 5th-generation tensor core (tcgen05: TMEM allocation, MMA, commit, loads),
// written from the PTX ISA description of those instructions; plus the
// workspace layout that the host API and every kernel agree on.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <map>
#include <set>
#include <utility>

namespace moe {

// Expert segments in the permuted buffers are padded to this many rows: the
// grouped GEMM's tile height, so a tile never straddles two experts.
constexpr int kSegRows = 128;
// Slots per dispatch-scan block (one thread per slot).
constexpr int kScanChunk = 1024;
// Tokens per router block.
constexpr int kRouterTokens = 32;
// Limits of this build (mirrored by MOE_MAX_EXPERTS / MOE_MAX_TOPK in moe.h).
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;

// Device error word bits (sticky until moe_last_device_status reads them).
enum : uint32_t {
    kErrTimeoutProducer = 1u,
    kErrTimeoutMma = 2u,
    kErrTimeoutEpilogue = 4u,
    kErrTimeoutDrain = 8u,
};

// Bounded waits give up after this long and flag kErrTimeout*.
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s

__host__ __device__ constexpr inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  A kernel launched with pdl = true may start while
// the previous kernel of its stream is still running; it must call griddep_wait()
// before reading anything earlier kernels wrote, and every such kernel calls it
// before exiting, so the completion of a grid implies that of all its predecessors.
// griddep_launch_dependents() lets the next kernel begin launching: it launches once
// every CTA of this grid has called it (or exited), so all of this grid's CTAs are
// resident by then and the early CTAs of the next kernel cannot starve them.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Kernels launched (or recorded into a CUDA graph under stream capture) by this
// library since it was loaded; read through moe_kernel_launches().
std::atomic<unsigned long long>& launch_counter();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 bool pdl, Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
    return e;
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device); later
// launches (including ones recorded into CUDA graphs) make no attribute call.
inline cudaError_t ensure_smem_limit(const void* kernel, size_t bytes)
{
    // the largest limit set so far per (kernel, device): kernels whose shared memory
    // depends on the layer's sizes raise it again when a later layer needs more
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({kernel, dev});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done[{kernel, dev}] = bytes;
    return e;
}
__host__ __device__ constexpr inline size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------------------
// Scalar helpers

// softplus(z) = ln(1 + e^z) as max(z, 0) + ln(1 + e^-|z|): no overflow for large z
__device__ __forceinline__ float softplus_f32(float z) { return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z))); }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte read-only load through the non-coherent path (data written by an earlier kernel).
__device__ __forceinline__ uint4 ld_stream(const uint4* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte vectors of a row as fp32: 8 bf16 or 4 fp32 elements.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void* p, float (&v)[8])
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(void* p, const float (&v)[8])
    {
        uint4 u;
        u.x = pack_bf16x2(v[0], v[1]);
        u.y = pack_bf16x2(v[2], v[3]);
        u.z = pack_bf16x2(v[4], v[5]);
        u.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void* p, float (&v)[4])
    {
        const float4 u = *reinterpret_cast<const float4*>(p);
        v[0] = u.x;
        v[1] = u.y;
        v[2] = u.z;
        v[3] = u.w;
    }
    __device__ static void store(void* p, const float (&v)[4])
    {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};


// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up
// (returns false) after kWaitTimeoutNs or as soon as *abort is set, so that no
// wait can spin forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of box {c0 (innermost), c1} into shared memory; completion is
// signalled on `bar` as transaction bytes.  c0 * element size must be a
// multiple of 16 bytes (callers pass multiples of 64 bf16 elements).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, uint64_t cache_policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
        "l"(cache_policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory)

// Allocate `ncols` TMEM columns (power of two >= 32); the TMEM address is
// written to shared memory.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row core groups 1024 B apart.
// Fields: start address >> 4 (bits 0-13), leading-dimension byte offset >> 4
// (bits 16-29, unused for swizzled K-major), stride-dimension byte offset >> 4
// (bits 32-45), descriptor version 1 (bits 46-47), swizzle mode 2 = 128-byte
// (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand tile stored with the
// 128-byte swizzle, as TMA writes a box of 64 MN-contiguous bf16 (128 B) by 64
// K-rows: one 8 KB block per 64 MN elements.  Inside a block, K-rows are 128 B
// apart and 8-row K groups 1024 B apart (stride-dimension offset); consecutive
// 64-element MN blocks are 8192 B apart (leading-dimension offset).  A K-step of
// 16 advances the start address by 16 rows = 2048 B.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(8192u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with A and/or B MN-major (bit 15: A, bit 16: B).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_major(int M, int N, bool a_mn, bool b_mn)
{
    return idesc_bf16_f32(M, N) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Each thread of the warp loads 32 consecutive fp32 columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// Each thread of the warp loads 16 consecutive fp32 columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Activations (fp32).  GELU(tanh), GELU(erf): Hendrycks & Gimpel; silu(z) = z / (1 + e^-z).

enum ActKind : int { kActNone = -1, kActRelu = 0, kActGeluTanh = 1, kActGeluErf = 2, kActSwiglu = 3 };

template <int ACT>
__device__ __forceinline__ float activate(float z)
{
    if constexpr (ACT == kActRelu) {
        return fmaxf(z, 0.0f);
    } else if constexpr (ACT == kActGeluTanh) {
        const float c = 0.7978845608028654f;  // sqrt(2/pi)
        return 0.5f * z * (1.0f + tanhf(c * (z + 0.044715f * z * z * z)));
    } else if constexpr (ACT == kActGeluErf) {
        return 0.5f * z * (1.0f + erff(z * 0.7071067811865476f));
    } else if constexpr (ACT == kActSwiglu) {
        return z / (1.0f + expf(-z));
    } else {
        return z;
    }
}

// Activations for epilogues whose result is rounded to bf16: the CUDA fast
// intrinsics (__expf, __fdividef; about 2 ulp of fp32) are far below bf16's
// rounding step and keep the unrolled epilogue small and branch-free.
//   silu(z) = z / (1 + e^-z);  tanh(u) = 1 - 2 / (1 + e^{2u}).
template <int ACT>
__device__ __forceinline__ float activate_bf16out(float z)
{
    if constexpr (ACT == kActSwiglu) {
        return __fdividef(z, 1.0f + __expf(-z));
    } else if constexpr (ACT == kActGeluTanh) {
        const float u = 0.7978845608028654f * (z + 0.044715f * z * z * z);
        return 0.5f * z * (2.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * u)));
    } else {
        return activate<ACT>(z);
    }
}

// Derivatives for the backward pass (fp32), from the definitions above:
//   silu'(z) = s (1 + z (1 - s)),  s = 1 / (1 + e^-z);
//   GELU(tanh)'(z) = (1 + th) / 2 + z (1 - th^2) c (1 + 3 a z^2) / 2,  th = tanh(c (z + a z^3));
//   GELU(erf)'(z) = Phi(z) + z phi(z).
__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float silu_grad_f32(float z)
{
    const float s = 1.0f / (1.0f + expf(-z));
    return s * (1.0f + z * (1.0f - s));
}
template <int ACT>
__device__ __forceinline__ float act_grad_f32(float z)
{
    if constexpr (ACT == kActRelu) {
        return z > 0.0f ? 1.0f : 0.0f;
    } else if constexpr (ACT == kActGeluTanh) {
        const float c = 0.7978845608028654f, a = 0.044715f;  // sqrt(2/pi)
        const float th = tanhf(c * (z + a * z * z * z));
        return 0.5f * (1.0f + th) + 0.5f * z * (1.0f - th * th) * c * (1.0f + 3.0f * a * z * z);
    } else if constexpr (ACT == kActGeluErf) {
        // 1/sqrt(2) and 1/sqrt(2 pi)
        return 0.5f * (1.0f + erff(z * 0.7071067811865476f)) + z * expf(-0.5f * z * z) * 0.3989422804014327f;
    } else {
        return silu_grad_f32(z);
    }
}

// ---------------------------------------------------------------------------
// Grouped GEMM problem description (shared by the tcgen05 and FFMA kernels).
//
// Groups are experts.  Group g owns rows [row_off(g), row_off(g) + rows(g)) of
// A and of the output; its M-tiles are numbered mtile_off[g] .. mtile_off[g+1]-1.
// Either the three arrays come from the dispatch scan (routed experts) or,
// when mtile_off == nullptr, there is one group of `fixed_rows` rows at row 0
// (shared experts over all tokens).
// B is the 2-D view [groups * b_rows_per_group, K] of a weight tensor; group g,
// K-segment s and output column n read B row
//   (b_group0 + g + s) * b_rows_per_group + n.
// A column of K-segment s is s * K + kk.  The output is [rows, ldo]; bias (if
// any) of output column n is sum_s bias[(b_group0 + g + s) * b_rows_per_group + n].
struct GroupedGemmArgs {
    const int* mtile_off;  // [G+1] device, or nullptr for one fixed group
    const int* row_off;    // [G] device padded row offsets
    const int* rows;       // [G] device valid rows per group
    int G;
    int fixed_rows;
    int N;                 // valid output columns per group
    int n_tiles;           // output column tiles per group
    int K;                 // reduction length of one K-segment
    int k_segments;
    int b_rows_per_group;
    int b_group0;
    void* out;
    int ldo;
    const void* bias;
    int a_rows_alloc;      // rows of A that exist (FFMA bounds)
    uint32_t* err;
    void* z1;              // tcgen05 kernel, training: pre-activations of the output, [rows, ldo], or nullptr
    void* z3;              // ... and the W3 half (SwiGLU)
};

}  // namespace moe
