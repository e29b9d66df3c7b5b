// noalloc.cu -- the LL all-pair allreduce for callers that cannot allocate
// device memory.
//
// sar_allreduce_ll needs a packet scratch of nranks x sar_ll_packet_bytes(count)
// bytes that the caller allocates.  Some callers cannot: code running inside a
// framework whose allocator owns all device memory, plugins with a fixed
// memory budget, or code paths where a cudaMalloc would synchronise the device
// or is not allowed at all.  This entry point takes the scratch from a fixed
// array compiled into the library instead, so the call itself allocates
// nothing.  MSCCL++ has no counterpart of this entry point.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library's device code reserves it and holds it until the process exits.  In
// host code its name is only a host-side stand-in, not a device address, so
// the address is looked up once per device with cudaGetSymbolAddress (with
// that device current) and passed to the kernels.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sar_internal.h"

namespace sar {
namespace {

// Packet scratch followed by one 256-byte slot holding the internal status
// word.  Static storage: zero when the module is loaded.
constexpr size_t kStatusSlot = 256;
static __device__ __align__(256) unsigned char g_ll_scratch[SAR_LL_NOALLOC_SCRATCH_BYTES + kStatusSlot];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
    std::mutex mu;
    std::atomic<unsigned char*> base{nullptr};   // device address of g_ll_scratch on this device
    std::atomic<uint32_t> epoch{0};               // last epoch used on this device
};

DeviceScratch g_dev[kMaxDevices];

// Device address of the scratch on the current device, looked up on first
// use.  Only a successful lookup is kept: after a failure (for example a first
// call made during a CUDA graph capture) the next call tries again.
cudaError_t scratch_base(int dev, unsigned char** out) {
    DeviceScratch& d = g_dev[dev];
    unsigned char* b = d.base.load(std::memory_order_acquire);
    if (b == nullptr) {
        std::lock_guard<std::mutex> lock(d.mu);
        b = d.base.load(std::memory_order_relaxed);
        if (b == nullptr) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_ll_scratch);
            if (e != cudaSuccess || p == nullptr) {
                // Reported here; cleared so that a later launch check does not
                // report it again.
                (void)cudaGetLastError();
                *out = nullptr;
                return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            }
            b = static_cast<unsigned char*>(p);
            d.base.store(b, std::memory_order_release);
        }
    }
    *out = b;
    return cudaSuccess;
}

bool supported(int n) { return n >= 1 && n <= SAR_MAX_RANKS; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The LL allreduce (pack, then unpack-reduce) on the fixed scratch, with a
// fresh epoch per call and device.  With d_status == nullptr the internal
// status word is cleared first and used, so that a timeout of an earlier call
// does not end this call's polls at once.
sar_status fixed_scratch_allreduce(const void* const* in, void* const* out, int nranks, size_t count,
                                   sar_dtype dtype, uint64_t max_spins, int32_t* d_status, cudaStream_t s) {
    if (!supported(nranks)) return SAR_ERR_UNSUPPORTED_NRANKS;
    if (dtype < SAR_BF16 || dtype > SAR_FP8_E4M3B15) return SAR_ERR_UNSUPPORTED_DTYPE;
    if (in == nullptr || out == nullptr || max_spins == 0) return SAR_ERR_INVALID_ARG;
    const size_t es = esize_of(dtype);
    if (count > (SIZE_MAX / 16) / es) return SAR_ERR_INVALID_ARG;
    // Each rank's packets start on a 256-byte boundary of the fixed array.
    const size_t stride = round256((count * es + 3) / 4 * 8);
    if (stride > SAR_LL_NOALLOC_SCRATCH_BYTES / static_cast<size_t>(nranks)) return SAR_ERR_INVALID_ARG;
    if (d_status != nullptr && reinterpret_cast<uintptr_t>(d_status) % 4 != 0) return SAR_ERR_MISALIGNED;
    if (count == 0) return SAR_OK;
    bool in16 = true, out16 = true;
    for (int r = 0; r < nranks; ++r) {
        if (in[r] == nullptr || out[r] == nullptr) return SAR_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(in[r]) % es != 0 || reinterpret_cast<uintptr_t>(out[r]) % es != 0)
            return SAR_ERR_MISALIGNED;
        in16 = in16 && reinterpret_cast<uintptr_t>(in[r]) % 16 == 0;
        out16 = out16 && reinterpret_cast<uintptr_t>(out[r]) % 16 == 0;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAR_ERR_CUDA;
    unsigned char* base = nullptr;
    if (scratch_base(dev, &base) != cudaSuccess || base == nullptr) return SAR_ERR_CUDA;

    // A fresh epoch per call on this device, so packets left in the shared
    // array by an earlier call never match.  After 2^32 - 1 calls the epoch
    // wraps: the packet area is zeroed again (epoch 0 means "never written").
    uint32_t epoch = g_dev[dev].epoch.fetch_add(1) + 1;
    if (epoch == 0) {
        if (cudaMemsetAsync(base, 0, SAR_LL_NOALLOC_SCRATCH_BYTES, s) != cudaSuccess) return SAR_ERR_CUDA;
        epoch = g_dev[dev].epoch.fetch_add(1) + 1;
    }
    int32_t* status = d_status;
    if (status == nullptr) {
        status = reinterpret_cast<int32_t*>(base + SAR_LL_NOALLOC_SCRATCH_BYTES);
        if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SAR_ERR_CUDA;
    }

    RankPtrs pack, unpack;
    std::memset(&pack, 0, sizeof(pack));
    std::memset(&unpack, 0, sizeof(unpack));
    for (int r = 0; r < nranks; ++r) {
        void* pk = base + static_cast<size_t>(r) * stride;
        pack.in[r] = in[r];
        pack.out[r] = pk;
        unpack.in[r] = pk;
        unpack.out[r] = out[r];
    }
    if (launch_ll_pack(nranks, pack, count * es, epoch, in16, s) != cudaSuccess) return SAR_ERR_CUDA;
    if (launch_ll_unpack_reduce(dtype, nranks, unpack, count, epoch, max_spins, status, out16, s) != cudaSuccess)
        return SAR_ERR_CUDA;
    return SAR_OK;
}

}  // namespace

unsigned char* testing_fixed_scratch(int dev, bool set_epoch, uint32_t last_epoch) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    if (set_epoch) g_dev[dev].epoch.store(last_epoch);
    return g_dev[dev].base.load();
}

}  // namespace sar

extern "C" SAR_API sar_status sar_allreduce_ll_noalloc(const void* const* in, void* const* out, int nranks,
                                                       size_t count, sar_dtype dtype, uint64_t max_spins,
                                                       int32_t* d_status, sar_stream_t stream) {
    return sar::fixed_scratch_allreduce(in, out, nranks, count, dtype, max_spins, d_status,
                                        reinterpret_cast<cudaStream_t>(stream));
}
