// dispatch_noalloc.cu -- allocation-free form of the dispatch scan.
//
// Some callers cannot allocate device memory at the point where they route
// tokens: a host engine that owns every byte of device memory through its own
// fixed pool and forbids libraries from calling cudaMalloc, or a
// latency-critical path that cannot pay cudaMalloc's implicit device
// synchronisation.  Such callers may also be unable to size and hand over the
// workspace that moe_workspace_size asks for.  moe_dispatch_positions_noalloc
// serves them: it computes the per-expert counts, the capacity drops and the
// permutation rows from the router's expert indices using only a scratch
// array that lives in this file as a static device variable.
//
// The scratch array exists once per device that loads the library and lives
// until the process exits.  Its size caps the problem at MOE_NOALLOC_MAX_SLOTS
// routed slots (T * k) and MOE_MAX_EXPERTS experts.  Every call on a device
// shares the same array and leaves its contents behind; the arrival counter
// that must start at zero is cleared at the start of each call.  Two calls
// whose kernels overlap on the GPU (e.g. on two streams) race on the array.
#include <mutex>

#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

constexpr int kNoallocMaxSlots = MOE_NOALLOC_MAX_SLOTS;
constexpr int kNoallocMaxChunks = (kNoallocMaxSlots + kScanChunk - 1) / kScanChunk;

// Byte offsets inside the scratch array (every region 256-byte aligned).
constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kOffDone = 0;
constexpr size_t kOffRank = 256;
constexpr size_t kOffHist = kOffRank + align256(sizeof(int32_t) * kNoallocMaxSlots);
constexpr size_t kOffBase = kOffHist + align256(sizeof(int32_t) * kNoallocMaxChunks * kMaxExperts);
constexpr size_t kOffKept = kOffBase + align256(sizeof(int32_t) * kNoallocMaxChunks * kMaxExperts);
constexpr size_t kOffRowOff = kOffKept + align256(sizeof(int32_t) * kMaxExperts);
constexpr size_t kOffKeptOff = kOffRowOff + align256(sizeof(int32_t) * kMaxExperts);
constexpr size_t kOffMtile = kOffKeptOff + align256(sizeof(int32_t) * kMaxExperts);
constexpr size_t kOffAux = kOffMtile + align256(sizeof(int32_t) * (kMaxExperts + 1));
constexpr size_t kScratchBytes = kOffAux + 256;  // about 1.03 MB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Per device: the device address of g_noalloc_scratch, looked up with that
// device current (the host-side symbol is not a device address).  Only a
// successful lookup is kept: a lookup that failed (for example one attempted
// during a stream capture, where loading the module is not allowed) is retried
// by the next call.
struct ScratchSlot {
    std::mutex mu;
    unsigned char* ptr = nullptr;
};
ScratchSlot g_slots[64];

cudaError_t scratch_for_current_device(unsigned char** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    ScratchSlot& s = g_slots[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.ptr == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // the failed lookup leaves no sticky error behind
            return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        }
        s.ptr = static_cast<unsigned char*>(p);
    }
    *out = s.ptr;
    return cudaSuccess;
}

// Token-order position of every slot: chunk base + rank inside the chunk.
__global__ void __launch_bounds__(256) k_positions_noalloc(DispatchArgs a)
{
    const long long n_slots = (long long)a.T * a.k;
    for (long long s = (long long)blockIdx.x * 256 + threadIdx.x; s < n_slots;
         s += (long long)gridDim.x * 256) {
        const int e = a.idx[s];
        const bool e_ok = e >= 0 && e < a.E;  // out-of-range indices are dropped
        const int c = (int)(s / kScanChunk);
        const int pos = e_ok ? a.chunk_base[(size_t)c * a.E + e] + a.local_rank[s] : 0;
        const bool keep = e_ok && (a.C < 0 || pos < a.C);
        a.dropped[s] = keep ? 0 : 1;
        a.perm_row[s] = keep ? a.kept_off[e] + pos : -1;
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_positions_noalloc(const moe_params_t* params,
                                                       const int32_t* expert_idx, int32_t* counts,
                                                       uint8_t* dropped, int32_t* perm_row,
                                                       void* stream)
{
    if (params == nullptr || expert_idx == nullptr || counts == nullptr || dropped == nullptr ||
        perm_row == nullptr)
        return MOE_ERR_INVALID_ARG;
    const moe_params_t& p = *params;
    if (p.T < 0 || p.E < 1 || p.E > MOE_MAX_EXPERTS || p.k < 1 || p.k > p.E || p.k > MOE_MAX_TOPK)
        return MOE_ERR_INVALID_ARG;
    if ((long long)p.T * p.k > kNoallocMaxSlots) return MOE_ERR_INVALID_ARG;  // scratch too small
    if (p.capacity_factor != p.capacity_factor) return MOE_ERR_INVALID_ARG;
    if (p.T == 0)  // an empty batch: no expert receives a token
        return cudaMemsetAsync(counts, 0, sizeof(int32_t) * p.E, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;

    unsigned char* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    int C = -1;
    if (p.capacity_factor > 0.0f) {
        const double c = (double)p.T * (double)p.capacity_factor / (double)p.E;
        C = c >= (double)p.T ? p.T : (int)c;  // floor of a non-negative value
    }
    DispatchArgs a{};
    a.idx = expert_idx;
    a.T = p.T;
    a.k = p.k;
    a.E = p.E;
    a.C = C;
    a.nchunks = (int)(((long long)p.T * p.k + kScanChunk - 1) / kScanChunk);
    a.n_router_blocks = 0;  // no balance statistic here
    a.psum_part = nullptr;
    a.local_rank = reinterpret_cast<int32_t*>(scratch + kOffRank);
    a.chunk_hist = reinterpret_cast<int32_t*>(scratch + kOffHist);
    a.chunk_base = reinterpret_cast<int32_t*>(scratch + kOffBase);
    a.scan_done = reinterpret_cast<unsigned*>(scratch + kOffDone);
    a.counts = counts;
    a.kept = reinterpret_cast<int32_t*>(scratch + kOffKept);
    a.row_off = reinterpret_cast<int32_t*>(scratch + kOffRowOff);
    a.kept_off = reinterpret_cast<int32_t*>(scratch + kOffKeptOff);
    a.mtile_off = reinterpret_cast<int32_t*>(scratch + kOffMtile);
    a.aux = reinterpret_cast<float*>(scratch + kOffAux);
    a.dropped = dropped;
    a.perm_row = perm_row;

    // the arrival counter of the scan must start at zero
    if (cudaMemsetAsync(scratch + kOffDone, 0, sizeof(unsigned), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_dispatch_scan_only(a, st) != cudaSuccess) return MOE_ERR_CUDA;
    const long long n_slots = (long long)p.T * p.k;
    const int grid = (int)((n_slots + 255) / 256 < 4096 ? (n_slots + 255) / 256 : 4096);
    return launch_kernel(k_positions_noalloc, dim3(grid), dim3(256), 0, st, false, a) == cudaSuccess ? MOE_OK
                                                                                          : MOE_ERR_CUDA;
}
