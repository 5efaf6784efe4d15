// Forward SpMM that allocates nothing: snk_forward_csr_noalloc.
//
// Who needs it: programs that hand the library no chance to allocate.  Some
// hosts own every byte of device memory through their own arena and forbid
// foreign cudaMalloc; in others cudaMalloc/cudaFree are off limits on the
// hot path because they synchronise the device and stall unrelated streams,
// or because the call runs where a failing allocation cannot be handled.
// Such callers cannot use snk_create (which allocates the topology
// workspace), so this entry point takes a ready CSR and keeps its own scratch
// in a fixed, statically sized device array that is part of the library
// image.
//
// The scratch array: the work partition (block boundaries, chunk and block
// descriptors), cross-block partial sums and per-row arrival counters of the
// merge-path kernel.  It is sized for at most kNaMaxBlocks blocks (one per
// SM) and kNaMaxOut output rows; larger requests are refused with
// SNK_ERR_LIMIT.  Every GPU that loads the library keeps this array for
// the life of the process.  All calls share it and it keeps the previous
// call's contents, so each call first clears the counters it uses, and two
// calls whose kernels overlap on the GPU (two streams, or two threads) race
// on it.
#include <mutex>

#include "snk_internal.cuh"

namespace snk {
namespace {

constexpr int kNaMaxBlocks = 512;                // blocks of the partition (one per SM)
constexpr int64_t kNaMaxOut = int64_t(1) << 19;  // 524,288 output rows
constexpr size_t kNaBndBytes = (size_t)(kNaMaxBlocks + 1) * sizeof(int32_t) + 12;  // 16-B padded
constexpr size_t kNaCdescBytes = (size_t)kNaMaxBlocks * kWarpsPerBlock * sizeof(int4);
constexpr size_t kNaBdescBytes = (size_t)kNaMaxBlocks * sizeof(BlockDesc);
constexpr size_t kNaPartBytes = (size_t)kNaMaxBlocks * 2 * kMaxBatchTile * sizeof(float);
constexpr size_t kNaCntBytes = (size_t)kNaMaxOut * sizeof(int32_t);
constexpr size_t kNaScratchBytes =
    kNaBndBytes + kNaCdescBytes + kNaBdescBytes + kNaPartBytes + kNaCntBytes;
constexpr int kNaMaxDevices = 64;

}  // namespace

// The scratch itself.  Host code must not use this name as a pointer: it is
// a host-side stand-in.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

namespace {

std::mutex g_mu;
void* g_addr[kNaMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_address(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kNaMaxDevices) return SNK_ERR_LIMIT;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SNK_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_addr[dev]);
    return SNK_OK;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace snk

using namespace snk;

extern "C" int snk_forward_csr_noalloc(int64_t out_features, int64_t in_features, int64_t nnz,
                                       const int32_t* row_ptr, const int32_t* cols,
                                       const float* values, const float* X, int64_t batch,
                                       const float* bias, float* Y, void* stream) {
    if (out_features < 1 || in_features < 1 || in_features > INT32_MAX || batch < 0 ||
        nnz < 0 || nnz > INT32_MAX)
        return SNK_ERR_ARG;
    if (out_features > kNaMaxOut) return SNK_ERR_LIMIT;
    if (batch == 0) return SNK_OK;
    if (!row_ptr || !X || !Y || (nnz > 0 && (!cols || !values))) return SNK_ERR_ARG;
    if (!aligned(values, 16) || !aligned(cols, 16) || !aligned(row_ptr, 4) || !aligned(X, 4) ||
        !aligned(Y, 4) || !aligned(bias, 4))
        return SNK_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;

    int dev = 0, num_sms = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        cudaGetLastError();
        return SNK_ERR_CUDA;
    }
    // the operand and the kernel's partial-sum slots must fit one block's
    // shared memory for the largest batch tile used (the first one), checked
    // before anything is queued
    const int64_t tile = batch < kMaxBatchTile ? batch : kMaxBatchTile;
    if (forward_csr_smem(in_features, batch_tile(tile)) > (size_t)max_smem) return SNK_ERR_LIMIT;

    // one block per SM, one chunk per warp
    const int n_blocks = num_sms;
    if (n_blocks > kNaMaxBlocks) return SNK_ERR_LIMIT;

    unsigned char* base = nullptr;
    int st = scratch_address(dev, &base);
    if (st != SNK_OK) return st;
    int32_t* bnd = reinterpret_cast<int32_t*>(base);
    int4* cdesc = reinterpret_cast<int4*>(base + kNaBndBytes);
    BlockDesc* bdesc = reinterpret_cast<BlockDesc*>(base + kNaBndBytes + kNaCdescBytes);
    float* part = reinterpret_cast<float*>(base + kNaBndBytes + kNaCdescBytes + kNaBdescBytes);
    int32_t* cnt =
        reinterpret_cast<int32_t*>(base + kNaBndBytes + kNaCdescBytes + kNaBdescBytes + kNaPartBytes);

    // the arrival counters must start at zero; the previous call's state is
    // not trusted
    if (cudaMemsetAsync(cnt, 0, (size_t)out_features * sizeof(int32_t), s) != cudaSuccess)
        return SNK_ERR_CUDA;
    st = build_partition(row_ptr, out_features, nnz, n_blocks, kWarpsPerBlock, bnd, cdesc, bdesc, s);
    if (st != SNK_OK) return st;
    return launch_forward_csr(values, cols, row_ptr, cdesc, bdesc, bnd, nnz, out_features,
                              in_features, n_blocks, X, batch, bias, Y, part, cnt, max_smem, s);
}
