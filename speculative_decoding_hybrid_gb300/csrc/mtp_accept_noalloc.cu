// mtp_greedy_accept_noalloc: the greedy accept of mtp_accept.cu for callers
// that cannot allocate device memory.
//
// Why: some callers have no device allocator of their own at the point where
// they accept drafts -- a plugin whose host engine owns all device memory and
// hands out none, or a latency-critical serving loop where a cudaMalloc (which
// may synchronise the whole device) is not acceptable.  This entry point takes
// the same inputs and outputs as mtp_greedy_accept but no workspace: its
// scratch (the per-split partial maxima) is a fixed array in the library's
// device image.
//
// Rules that follow from a shared, fixed scratch:
//  * The array holds kNoAllocPartials 64-bit keys (512 KiB) and lives on every
//    device that loads the library until the process exits.  A request needing
//    more (mtp_accept_workspace_bytes(row_capacity, vocab) > 512 KiB) is
//    refused with GDN_ERR_WORKSPACE before anything is launched.
//  * Every call uses the same array and it keeps the previous call's contents.
//    Nothing in it needs to start at zero: each call writes every entry it
//    later reads.  Calls whose kernels overlap on the GPU (different streams,
//    no ordering between them) race on the array and must not be issued.
//  * The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture.  No call allocates or frees memory.
//    The cached address is not refreshed: after a cudaDeviceReset of that
//    device it is stale, and the entry point must not be called there again.
#include <mutex>

#include "common.cuh"

int gdn_accept_launch(int32_t B, int32_t row_capacity, const int32_t *cu_rows, const gdn_bf16 *logits,
                      int64_t vocab, int64_t row_stride, const int32_t *tokens, int32_t *argmax,
                      int32_t *accept_len, int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                      void *workspace, size_t workspace_bytes, uint32_t *dev_status, cudaStream_t st);

namespace {

constexpr size_t kNoAllocPartials = 65536;
static __device__ __align__(256) unsigned long long g_accept_scratch[kNoAllocPartials];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_accept_scratch, per device

int scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" int mtp_greedy_accept_noalloc(int32_t B, int32_t row_capacity, const int32_t *cu_rows,
                                         const gdn_bf16 *logits, int64_t vocab, int64_t row_stride,
                                         const int32_t *tokens, int32_t *argmax, int32_t *accept_len,
                                         int32_t *bonus, int32_t *out_tokens, mtp_stats *stats,
                                         uint32_t *dev_status, void *stream) {
    if (B < 0 || row_capacity < 0 || vocab <= 0) return GDN_ERR_ARG;
    if (mtp_accept_workspace_bytes(row_capacity, vocab) > sizeof(g_accept_scratch)) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
    return gdn_accept_launch(B, row_capacity, cu_rows, logits, vocab, row_stride, tokens, argmax, accept_len, bonus,
                             out_tokens, stats, scratch, sizeof(g_accept_scratch), dev_status,
                             static_cast<cudaStream_t>(stream));
}
