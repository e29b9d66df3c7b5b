// ll_packets.cuh -- the LL packet: 8 bytes, a 4-byte payload word and the
// 4-byte epoch flag above it, always written and read by one
// single-copy-atomic 8-byte access so that a reader that sees the flag also
// sees the payload.  Vector accesses (16 or 32 bytes) are sets of such 8-byte
// element accesses.  volatile keeps every poll a fresh read.
#pragma once

#include <cstdint>

namespace sar {

__device__ __forceinline__ void ld_packets2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint64_t ld_packet(const uint64_t* p) {
    uint64_t a;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void st_packet(uint64_t* p, uint64_t a) {
    asm volatile("st.volatile.global.u64 [%0], %1;" :: "l"(p), "l"(a) : "memory");
}
__device__ __forceinline__ void st_packets2(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" :: "l"(p), "l"(a), "l"(b) : "memory");
}
// Four packets in one 32-byte access (sm_100 and later); p must be 32-byte aligned.
__device__ __forceinline__ void st_packets4(uint64_t* p, uint64_t a, uint64_t b, uint64_t c, uint64_t d) {
    asm volatile("st.volatile.global.v4.u64 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "l"(a), "l"(b), "l"(c), "l"(d) : "memory");
}

__device__ __forceinline__ uint64_t make_packet(uint32_t payload, uint32_t epoch) {
    return static_cast<uint64_t>(payload) | (static_cast<uint64_t>(epoch) << 32);
}
__device__ __forceinline__ uint32_t packet_flag(uint64_t p) { return static_cast<uint32_t>(p >> 32); }
__device__ __forceinline__ uint32_t packet_payload(uint64_t p) { return static_cast<uint32_t>(p); }

// Payload word w of a byte buffer of nbytes: bytes 4w..4w+3, little-endian,
// zero past the end (the padding of the last packet).
__device__ __forceinline__ uint32_t payload_word(const unsigned char* b, size_t nbytes, size_t w) {
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k)
        if (4 * w + k < nbytes) v |= static_cast<uint32_t>(b[4 * w + k]) << (8 * k);
    return v;
}

// The caller's status word, read fresh on every call (a poll that has to wait
// checks whether another thread has already given up).
__device__ __forceinline__ int32_t ld_status_word(const int32_t* s) {
    int32_t v;
    asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(s) : "memory");
    return v;
}

// One payload word of a result, stored to an output without allocating in L1.
__device__ __forceinline__ void st_stream_word(uint32_t* p, uint32_t v) {
    asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

}  // namespace sar
