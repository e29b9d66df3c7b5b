// noalloc_wrap_check.cu -- the epoch wrap of the library's fixed LL scratch,
// driven from a test program that links libsar's object files (the hook that
// sets the epoch counter is internal and not exported by libsar.so).
//
//   1. An LL allreduce through sar_allreduce_ll_noalloc with 64K fp32 per rank
//      fills the fixed array with packets of some epoch.
//   2. The per-device epoch counter is set to 2^32 - 1, so the next call wraps:
//      it must zero the array, then use epoch 1.  That call (1000 fp32 per
//      rank) must equal the rsag allreduce, its own packets must carry epoch 1,
//      and every byte past its packets must be zero (the big call's packets
//      would still be there without the clear).
//   3. One more call (64K per rank) uses epoch 2 and equals the rsag allreduce.
// Prints OK and exits 0 on success.
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "sar.h"

namespace sar {
unsigned char* testing_fixed_scratch(int dev, bool set_epoch, uint32_t last_epoch);
}

#define CK(x)                                                                     \
    do {                                                                          \
        cudaError_t e_ = (x);                                                     \
        if (e_ != cudaSuccess) {                                                  \
            std::printf("%s: %s\n", #x, cudaGetErrorString(e_));                  \
            return 1;                                                             \
        }                                                                         \
    } while (0)
#define SK(x)                                                                     \
    do {                                                                          \
        sar_status s_ = (x);                                                      \
        if (s_ != SAR_OK) {                                                       \
            std::printf("%s: %s\n", #x, sar_status_string(s_));                   \
            return 1;                                                             \
        }                                                                         \
    } while (0)

constexpr int kRanks = 8;
constexpr size_t kBig = 65536, kSmall = 1000;

static int same(const std::vector<void*>& a, const std::vector<void*>& b, size_t count, const char* what) {
    std::vector<uint32_t> ha(count), hb(count);
    for (int j = 0; j < kRanks; ++j) {
        if (cudaMemcpy(ha.data(), a[j], count * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
            cudaMemcpy(hb.data(), b[j], count * 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
            std::printf("%s: copy failed\n", what);
            return 0;
        }
        if (std::memcmp(ha.data(), hb.data(), count * 4) != 0) {
            std::printf("%s: out[%d] differs\n", what, j);
            return 0;
        }
    }
    return 1;
}

int main() {
    CK(cudaSetDevice(0));
    std::vector<void*> in(kRanks), got(kRanks), want(kRanks);
    std::vector<float> h(kBig);
    for (int r = 0; r < kRanks; ++r) {
        for (size_t i = 0; i < kBig; ++i) h[i] = static_cast<float>(static_cast<int>((r * 7 + i * 3) % 17) - 8);
        CK(cudaMalloc(&in[r], kBig * 4));
        CK(cudaMalloc(&got[r], kBig * 4));
        CK(cudaMalloc(&want[r], kBig * 4));
        CK(cudaMemcpy(in[r], h.data(), kBig * 4, cudaMemcpyHostToDevice));
    }
    int32_t* st = nullptr;
    CK(cudaMalloc(&st, 4));
    CK(cudaMemset(st, 0, 4));

    // 1. Fill the array.
    SK(sar_allreduce_ll_noalloc(in.data(), got.data(), kRanks, kBig, SAR_FP32, 1u << 20, st, nullptr));
    SK(sar_allreduce(in.data(), want.data(), kRanks, kBig, SAR_FP32, SAR_ALGO_RSAG, nullptr));
    CK(cudaDeviceSynchronize());
    if (!same(got, want, kBig, "first call")) return 1;
    unsigned char* base = sar::testing_fixed_scratch(0, true, 0xFFFFFFFFu);
    if (base == nullptr) {
        std::printf("fixed scratch not set up\n");
        return 1;
    }

    // 2. The wrapping call.
    SK(sar_allreduce_ll_noalloc(in.data(), got.data(), kRanks, kSmall, SAR_FP32, 1u << 20, st, nullptr));
    SK(sar_allreduce(in.data(), want.data(), kRanks, kSmall, SAR_FP32, SAR_ALGO_RSAG, nullptr));
    CK(cudaDeviceSynchronize());
    if (!same(got, want, kSmall, "wrapping call")) return 1;
    const size_t stride_small = (kSmall * 8 + 255) / 256 * 256, stride_big = kBig * 8;
    std::vector<uint32_t> words(kRanks * stride_big / 4);
    CK(cudaMemcpy(words.data(), base, words.size() * 4, cudaMemcpyDeviceToHost));
    for (int r = 0; r < kRanks; ++r) {
        const uint32_t* slot = words.data() + r * stride_small / 4;
        for (size_t w = 0; w < kSmall; ++w)
            if (slot[2 * w + 1] != 1u) {
                std::printf("rank %d packet %zu has flag %u, want 1\n", r, w, slot[2 * w + 1]);
                return 1;
            }
        for (size_t b = kSmall * 8 / 4; b < stride_small / 4; ++b)
            if (slot[b] != 0u) {
                std::printf("rank %d: byte %zu past the packets is not zero\n", r, 4 * b);
                return 1;
            }
    }
    for (size_t b = kRanks * stride_small / 4; b < words.size(); ++b)
        if (words[b] != 0u) {
            std::printf("byte %zu past the wrapping call's packets is not zero\n", 4 * b);
            return 1;
        }

    // 3. The next call uses epoch 2.
    SK(sar_allreduce_ll_noalloc(in.data(), got.data(), kRanks, kBig, SAR_FP32, 1u << 20, st, nullptr));
    SK(sar_allreduce(in.data(), want.data(), kRanks, kBig, SAR_FP32, SAR_ALGO_RSAG, nullptr));
    CK(cudaDeviceSynchronize());
    if (!same(got, want, kBig, "call after the wrap")) return 1;
    uint32_t flag = 0;
    CK(cudaMemcpy(&flag, base + 4, 4, cudaMemcpyDeviceToHost));
    if (flag != 2u) {
        std::printf("epoch after the wrap is %u, want 2\n", flag);
        return 1;
    }
    if (sar_read_device_status(st, nullptr) != SAR_OK) {
        std::printf("status not OK\n");
        return 1;
    }
    std::printf("OK\n");
    return 0;
}
