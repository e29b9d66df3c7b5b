// ll_coop.cuh -- the LL all-pair allreduce in one launch: the kernels shared
// by sar_allreduce_ll_fused (ll_fused.cu) and sar_allreduce_ll_writeback
// (ll_writeback.cu).  Calls up to a size limit (direct and multi-destination
// write-backs) run the sliced form further down, in which every block plays
// all ranks for one slice of the packets; the others run the cooperative form:
//
// mscclpp commit history, the allreduce_allpair_packet fix: the same thread
// block sends, reduces and writes back.  Every block of simulated rank r
//   A. packs its share of rank r's input into pkts[r] (the send): 16 input
//      bytes per thread and step, as one 32-byte packet store when every
//      packet buffer is 32-byte aligned, else two 16-byte stores;
//   B. polls its share of rank r's packet chunk in all N packet buffers (the
//      packets are written by other blocks of the same launch), one packet
//      index per thread and step, reduces in rank order and rounds once;
//   C. writes the result back, in one of three ways (template WB):
//        kDirect     - plain stores from registers to all N outputs;
//        kPacketsAll - as flagged result packets into `res`; then a block of
//                      rank r polls the result packets of chunk (r + 1) mod N
//                      and writes each one, read once, to all N outputs (the
//                      read-once, write-to-several-destinations fusion of the
//                      commit history's ReadPutPacket change);
//        kPacketsOwn - as result packets; then every rank j polls all result
//                      packets, starting with its own chunk, and writes its
//                      own output only.
//      Result packets are read 4 at a time (16-byte loads); rank chunks are
//      whole groups of 4 packets, so a group never spans two chunks.
// Each 8-byte packet is one single-copy-atomic store and load, so a flag that
// matches the epoch guarantees its payload; a stale flag means "not arrived".
// Every poll is bounded.  In this form blocks wait on one another, so the
// launch is cooperative: the runtime makes every block co-resident or refuses
// the launch.
//
// Epochs: the caller's, or a device counter (commit history, the flag buffer
// change: one flag buffer shared by the algorithms) that every launch advances
// by itself (take_ticket), so a replayed CUDA graph gets a fresh epoch.
#pragma once

#include <algorithm>
#include <atomic>

#include "ll_packets.cuh"
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace llc {

enum WriteBack { kDirect = 0, kPacketsAll = 1, kPacketsOwn = 2 };

constexpr unsigned kMaxSleepNs = 1024;
constexpr uint64_t kSpinPolls = 16;
// Input vectors a send thread loads before it stores their packets.
constexpr int kSendBatch = 4;


// Wait until packets w[0..n) (already loaded) carry `epoch`; false when this
// thread gave up or saw another thread give up.
template <int N>
__device__ __forceinline__ bool poll(const uint64_t* src, uint32_t epoch, uint64_t max_spins, int32_t* status,
                                     uint64_t (&w)[N]) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        bool ready = true;
#pragma unroll
        for (int i = 0; i < N; ++i) ready = ready && packet_flag(w[i]) == epoch;
        if (ready) return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        // The packets come from other blocks of this launch, usually within a
        // few hundred cycles: re-read at once for the first polls, then back
        // off (measured: 3-15% faster from 4 KiB per rank up than sleeping
        // from the first miss).  Only a thread that has started to back off
        // looks at the shared status word.
        if (spin >= kSpinPolls) {
            if (ld_status_word(status) != 0) return false;
            __nanosleep(ns);
            if (ns < kMaxSleepNs) ns *= 2;
        }
        if constexpr (N == 4) {
            ld_packets2(src, w[0], w[1]);
            ld_packets2(src + 2, w[2], w[3]);
        } else {
            w[0] = ld_packet(src);
        }
    }
}

// Wait until packet w of every rank k0 .. k0 + WIN - 1 (below n; already
// loaded into pk) carries `epoch`.  Every stale packet of the window is
// re-read in the same step, so a step costs one memory round trip whatever
// the rank count (re-reading the ranks one after another cost one round trip
// per stale rank).  False when this thread gave up or saw another give up.
template <int WIN, int NR>
__device__ __forceinline__ bool poll_window(uint64_t* const* pkts, int k0, int n, size_t w, uint32_t epoch,
                                            uint64_t max_spins, int32_t* status, uint64_t (&pk)[WIN]) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        bool ready = true;
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
            ready = ready && packet_flag(pk[k]) == epoch;
        }
        if (ready) return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        if (spin >= kSpinPolls) {
            if (ld_status_word(status) != 0) return false;
            __nanosleep(ns);
            if (ns < kMaxSleepNs) ns *= 2;
        }
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
            if (packet_flag(pk[k]) != epoch) pk[k] = ld_packet(pkts[k0 + k] + w);
        }
    }
}

// The device epoch counter: one uint64 whose bits kTicketBits.. count the
// launches that used it and whose low bits are zero between launches.  Every
// block of a launch adds to it once, block (0, 0) 2^kTicketBits - (blocks - 1)
// and every other block 1, so one launch adds exactly 2^kTicketBits.  The
// launches of one counter run one after another (stream order), so the value
// each block gets back lies in [k * 2^kTicketBits, (k + 1) * 2^kTicketBits)
// for the k-th launch whatever the order of the adds, and every block derives
// the same epoch (k mod (2^32 - 1)) + 1 from it: never 0, and consecutive
// launches always differ.  No block waits for another and nothing is written
// at the end of the launch.
constexpr int kTicketBits = 20;
__device__ __forceinline__ uint32_t take_ticket(uint64_t* ctrl) {
    const uint64_t blocks = static_cast<uint64_t>(gridDim.x) * gridDim.y;
    const uint64_t inc = (blockIdx.x == 0 && blockIdx.y == 0) ? (uint64_t(1) << kTicketBits) - (blocks - 1) : 1;
    uint64_t old;
    asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(ctrl), "l"(inc) : "memory");
    return static_cast<uint32_t>((old >> kTicketBits) % 0xFFFFFFFFull) + 1;
}

struct LLArgs {
    RankPtrs data;                   // in[r]: inputs, out[j]: outputs
    uint64_t* pkts[SAR_MAX_RANKS];   // send packet buffers
    uint64_t* res;                   // result packet buffer (packet write-back only)
};

// Raw element e of a payload word, stored as bits (no conversion).
template <int DT> __device__ __forceinline__ void store_bits(void* base, size_t i, uint32_t word, int e) {
    constexpr int ES = Elem<DT>::kSize;
    if constexpr (ES == 4) static_cast<uint32_t*>(base)[i] = word;
    else if constexpr (ES == 2) static_cast<uint16_t*>(base)[i] = static_cast<uint16_t>(word >> (16 * e));
    else static_cast<unsigned char*>(base)[i] = static_cast<unsigned char>(word >> (8 * e));
}

// Phase A: rank r's input -> pkts[r].  x0 is this thread's first input vector,
// already loaded when tid < nbytes / 16 and the input is 16-byte aligned.
__device__ __forceinline__ void send(const LLArgs& a, size_t nbytes, uint32_t epoch, bool in16, bool pk32,
                                     size_t tid, size_t stride, const uint4& x0) {
    const int r = blockIdx.y;
    const size_t npk = (nbytes + 3) / 4;
    uint64_t* mine = a.pkts[r];
    const size_t nfull = nbytes / 16;
    if (in16) {
        const uint4* src = static_cast<const uint4*>(a.data.in[r]);
        // A thread's vectors q0, q0 + stride, ... are loaded kSendBatch at a
        // time before any of them is stored (the packet stores are ordered
        // memory operations that later loads may not pass), so one memory
        // round trip covers a batch.
        for (size_t q0 = tid; q0 < nfull; q0 += kSendBatch * stride) {
            uint4 x[kSendBatch];
#pragma unroll
            for (int u = 0; u < kSendBatch; ++u) {
                const size_t q = q0 + u * stride;
                x[u] = make_uint4(0, 0, 0, 0);
                if (u == 0 && q0 == tid) x[u] = x0;
                else if (q < nfull) x[u] = ld_stream(src + q);
            }
#pragma unroll
            for (int u = 0; u < kSendBatch; ++u) {
                const size_t q = q0 + u * stride;
                if (q >= nfull) break;
                const uint64_t p0 = make_packet(x[u].x, epoch), p1 = make_packet(x[u].y, epoch);
                const uint64_t p2 = make_packet(x[u].z, epoch), p3 = make_packet(x[u].w, epoch);
                if (pk32) {
                    st_packets4(mine + 4 * q, p0, p1, p2, p3);
                } else {
                    st_packets2(mine + 4 * q, p0, p1);
                    st_packets2(mine + 4 * q + 2, p2, p3);
                }
            }
        }
    }
    const unsigned char* b = static_cast<const unsigned char*>(a.data.in[r]);
    for (size_t w = (in16 ? 4 * nfull : 0) + tid; w < npk; w += stride) {
        st_packet(mine + w, make_packet(payload_word(b, nbytes, w), epoch));
    }
}

// Phase B (+ C for kDirect): reduce rank r's chunk of packets
// [r*chunk, (r+1)*chunk), one packet index per thread and iteration.  False
// when a poll gave up.
template <int DT, int NR, int WB>
__device__ __forceinline__ bool reduce(const LLArgs& a, int n_rt, size_t count, size_t nbytes, size_t chunk,
                                       uint32_t epoch, uint64_t max_spins, int32_t* status, bool out16, size_t tid,
                                       size_t stride) {
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR == 0 ? 4 : (NR < 8 ? NR : 8);
    const int n = ranks<NR>(n_rt);
    const size_t npk = (nbytes + 3) / 4;
    const size_t wb = static_cast<size_t>(blockIdx.y) * chunk;
    const size_t we = min(npk, wb + chunk);
    for (size_t w = wb + tid; w < we; w += stride) {
        float acc[EP];
#pragma unroll 1
        for (int k0 = 0; k0 < n; k0 += WIN) {
            uint64_t pk[WIN];
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (NR == 0 && k0 + k >= n) break;
                pk[k] = ld_packet(a.pkts[k0 + k] + w);
            }
            if (!poll_window<WIN, NR>(a.pkts, k0, n, w, epoch, max_spins, status, pk)) return false;
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (NR == 0 && k0 + k >= n) break;
                float x[EP];
                widen_word<DT>(packet_payload(pk[k]), x);
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[e] = (k0 + k == 0) ? x[e] : __fadd_rn(acc[e], x[e]);
            }
        }
        if constexpr (WB != kDirect) {
            // Elements past the end are zero bits, as in the send's padding.
            float xs[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) xs[e] = (w * EP + e < count) ? acc[e] : 0.0f;
            st_packet(a.res + w, make_packet(narrow_word<DT>(xs), epoch));
        } else if (out16 && 4 * (w + 1) <= nbytes) {
            const uint32_t y = narrow_word<DT>(acc);
#pragma unroll
            for (int j = 0; j < n; ++j) st_stream_word(static_cast<uint32_t*>(a.data.out[j]) + w, y);
        } else {
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const size_t i = w * EP + e;
                if (i < count)
                    for (int j = 0; j < n; ++j) store_elem<DT>(a.data.out[j], i, acc[e]);
            }
        }
    }
    return true;
}

// Phase C for the packet write-backs: poll the result packets [wb, we) (wb a
// multiple of 4), 4 at a time (step `stride` groups), and store their payload
// to outputs [j0, j1).
template <int DT>
__device__ __forceinline__ bool unpack_results(const LLArgs& a, size_t count, size_t nbytes, size_t wb, size_t we,
                                               size_t rot, int j0, int j1, uint32_t epoch, uint64_t max_spins,
                                               int32_t* status, bool out16, size_t tid, size_t stride) {
    constexpr int EP = PerWord<DT>::kN;
    const size_t g0 = wb / 4, ng = (we + 3) / 4 - g0;
    for (size_t i = tid; i < ng; i += stride) {
        size_t q = g0 + i + rot;
        if (q >= g0 + ng) q -= ng;
        if (16 * (q + 1) <= nbytes) {
            uint64_t w[4];
            ld_packets2(a.res + 4 * q, w[0], w[1]);
            ld_packets2(a.res + 4 * q + 2, w[2], w[3]);
            if (!poll<4>(a.res + 4 * q, epoch, max_spins, status, w)) return false;
            const uint4 y = make_uint4(packet_payload(w[0]), packet_payload(w[1]), packet_payload(w[2]),
                                       packet_payload(w[3]));
            if (out16) {
                for (int j = j0; j < j1; ++j) st_stream(static_cast<uint4*>(a.data.out[j]) + q, y);
            } else {
                const uint32_t words[4] = {y.x, y.y, y.z, y.w};
                for (int j = j0; j < j1; ++j)
#pragma unroll
                    for (int m = 0; m < 4; ++m)
#pragma unroll
                        for (int e = 0; e < EP; ++e) store_bits<DT>(a.data.out[j], (4 * q + m) * EP + e, words[m], e);
            }
        } else {
            const size_t wend = min(we, 4 * q + 4);
            for (size_t wi = 4 * q; wi < wend; ++wi) {
                uint64_t pk[1] = {ld_packet(a.res + wi)};
                if (!poll<1>(a.res + wi, epoch, max_spins, status, pk)) return false;
                const uint32_t word = packet_payload(pk[0]);
                for (int j = j0; j < j1; ++j)
#pragma unroll
                    for (int e = 0; e < EP; ++e)
                        if (wi * EP + e < count) store_bits<DT>(a.data.out[j], wi * EP + e, word, e);
            }
        }
    }
    return true;
}

template <int DT, int NR, int WB>
__global__ void __launch_bounds__(kThreads)
coop_kernel(const LLArgs a, int n_rt, size_t count, size_t nbytes, size_t chunk, uint32_t host_epoch,
            uint64_t* ctrl, uint64_t max_spins, int32_t* status, bool in16, bool out16, bool pk32) {
    pdl_wait();
    const size_t tid = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    // The first input vector is loaded before the epoch is known, so that
    // load and the control-block read are in flight together.
    uint4 x0 = make_uint4(0, 0, 0, 0);
    if (in16 && tid < nbytes / 16) x0 = ld_stream(static_cast<const uint4*>(a.data.in[blockIdx.y]) + tid);
    __shared__ uint32_t s_epoch;
    if (threadIdx.x == 0) {
        uint32_t e = host_epoch;
        if (ctrl != nullptr) e = take_ticket(ctrl);
        s_epoch = e;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    const int n = ranks<NR>(n_rt);
    send(a, nbytes, epoch, in16, pk32, tid, stride, x0);
    bool ok = reduce<DT, NR, WB>(a, n_rt, count, nbytes, chunk, epoch, max_spins, status, out16, tid, stride);
    const size_t npk = (nbytes + 3) / 4;
    if constexpr (WB == kPacketsAll) {
        // Chunk (r + 1) mod N, reduced by other blocks: each result packet is
        // read once and written to every output.
        const size_t c = (static_cast<size_t>(blockIdx.y) + 1) % n;
        const size_t wb = c * chunk, we = min(npk, wb + chunk);
        if (ok && wb < we)
            unpack_results<DT>(a, count, nbytes, wb, we, 0, 0, n, epoch, max_spins, status, out16, tid, stride);
    } else if constexpr (WB == kPacketsOwn) {
        // Rank j reads every result packet and writes its own output, starting
        // with its own chunk (reduced by this rank's blocks just before).
        const int j = blockIdx.y;
        const size_t ng = (npk + 3) / 4, rot = min(ng, j * chunk / 4);
        if (ok)
            unpack_results<DT>(a, count, nbytes, 0, npk, rot == ng ? 0 : rot, j, j + 1, epoch, max_spins, status,
                               out16, tid, stride);
    }

}

// ---------------------------------------------------------------------------
// Sliced form: block b plays every rank for packets
// [b*SP, (b+1)*SP) of the buffers (SP = PPT*kSliceThreads packets per rank),
// so no block waits for another and the launch needs no co-residency.  In a
// slice:
//   A. item (k, g) packs input vector g of the slice of rank k into pkts[k]
//      (items spread over the threads, rotated by a warp per rank, so the
//      packets a warp polls come from other warps; the loads of up to 8
//      items are issued before their packet stores);
//   B. thread t polls packets PPT*t .. PPT*t+PPT-1 of every rank (windows of
//      up to 8 ranks polled together), adds in rank order, rounds once;
//   C. kDirect: plain stores of the result to all N outputs; kPacketsAll: the
//      result as flagged packets into `res`, then thread t polls the result
//      packets another warp wrote and writes each, read once, to all N
//      outputs; kPacketsOwn: the same result packets, then item (j, q) has
//      output rank j read result group q (4 packets) and write output j, the
//      items spread over the threads.
// The packet and result-packet images are those of the cooperative form.
// Measured against it (8 ranks fp32, CUDA graph, us per call, cooperative /
// sliced): direct write-back 1 KiB 2.30 / 1.90, 64 KiB 2.89 / 2.18, 256 KiB
// 3.72 / 3.04, 1 MiB 6.44 / 6.74; multi-destination packet write-back 1 KiB
// 2.73 / 2.14, 256 KiB 4.56 / 3.48, 1 MiB 8.28 / 7.59, 4 MiB 26.6 / 44.2;
// per-output packet write-back (result packets read once per output rank,
// the (rank, group) items spread over the threads) 1 KiB 2.87 / 2.59,
// 16 KiB 3.24 / 2.84, 256 KiB 4.48 / 4.14, 1 MiB 8.16 / 8.90.  4 packets per
// thread in the reduce (16-byte stores, 128 registers) was slower at 1 MiB
// (7.38 us direct).
// ---------------------------------------------------------------------------
constexpr int kSliceThreads = 128;
constexpr int kSlicePackets = 1;          // packets per thread and rank
// Largest bytes per rank that run sliced (measured crossovers, 8 ranks fp32).
constexpr size_t kSliceDirectMaxBytes = size_t(256) << 10;
constexpr size_t kSliceMultiDestMaxBytes = size_t(1) << 20;
constexpr size_t kSliceOwnMaxBytes = size_t(256) << 10;

template <int N>
__device__ __forceinline__ bool poll_slot(const uint64_t* src, int m_live, uint32_t epoch, uint64_t max_spins,
                                          int32_t* status, uint64_t (&w)[N]) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        bool ready = true;
#pragma unroll
        for (int m = 0; m < N; ++m) ready = ready && (m >= m_live || packet_flag(w[m]) == epoch);
        if (ready) return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        if (spin >= kSpinPolls) {
            if (ld_status_word(status) != 0) return false;
            __nanosleep(ns);
            if (ns < kMaxSleepNs) ns *= 2;
        }
#pragma unroll
        for (int m = 0; m < N; ++m)
            if (m < m_live && packet_flag(w[m]) != epoch) w[m] = ld_packet(src + m);
    }
}

// Result packets [w, w + m_live) of one thread (m_live <= PPT): load them,
// then (finish_slot) poll until they carry the epoch and store their payloads
// to outputs [j0, j1).
template <int PPT>
__device__ __forceinline__ void load_slot(const uint64_t* res, size_t w, int m_live, uint64_t (&r)[PPT]) {
    if (PPT == 4 && m_live >= 4) {
        ld_packets2(res + w, r[0], r[PPT > 1 ? 1 : 0]);
        ld_packets2(res + w + 2, r[PPT > 2 ? 2 : 0], r[PPT > 3 ? 3 : 0]);
    } else {
#pragma unroll
        for (int m = 0; m < PPT; ++m) r[m] = m < m_live ? ld_packet(res + w + m) : 0;
    }
}

template <int DT, int PPT>
__device__ __forceinline__ bool finish_slot(const LLArgs& a, size_t count, size_t nbytes, size_t w, int m_live, int j0,
                                            int j1, uint32_t epoch, uint64_t max_spins, int32_t* status, bool out16,
                                            uint64_t (&r)[PPT]) {
    constexpr int EP = PerWord<DT>::kN;
    if (!poll_slot<PPT>(a.res + w, m_live, epoch, max_spins, status, r)) return false;
    if (out16 && m_live >= PPT && 4 * (w + PPT) <= nbytes) {
        if constexpr (PPT == 4) {
            const uint4 y = make_uint4(packet_payload(r[0]), packet_payload(r[1]), packet_payload(r[2]),
                                       packet_payload(r[3]));
            for (int j = j0; j < j1; ++j) st_stream(static_cast<uint4*>(a.data.out[j]) + w / 4, y);
        } else {
#pragma unroll
            for (int m = 0; m < PPT; ++m)
                for (int j = j0; j < j1; ++j)
                    st_stream_word(static_cast<uint32_t*>(a.data.out[j]) + w + m, packet_payload(r[m]));
        }
    } else {
        for (int m = 0; m < PPT && m < m_live; ++m)
            for (int j = j0; j < j1; ++j)
#pragma unroll
                for (int e = 0; e < EP; ++e)
                    if ((w + m) * EP + e < count) store_bits<DT>(a.data.out[j], (w + m) * EP + e, packet_payload(r[m]), e);
    }
    return true;
}

// Phase A of the sliced form, in windows of up to 8 items per thread: item
// it = threadIdx.x + (u0 + u) * CT is input vector g of rank k of the slice
// starting at packet w0 (np packets).  slice_load issues the loads of a
// window, slice_store writes their packets.
template <int G, int CT>
__device__ __forceinline__ void slice_load(const LLArgs& a, int n, size_t nbytes, bool in16, size_t w0, int np, int u0,
                                           uint32_t (&x)[8][4]) {
    const int items = n * G;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int it = threadIdx.x + (u0 + u) * CT;
        const int k = it / G, g = (it + 32 * k) % G;
        if (it >= items || 4 * g >= np) continue;
        const size_t w = w0 + 4 * static_cast<size_t>(g);
        const unsigned char* src = static_cast<const unsigned char*>(a.data.in[k]);
        if (in16 && 4 * (w + 4) <= nbytes) {
            const uint4 q = ld_stream(reinterpret_cast<const uint4*>(src) + w / 4);
            x[u][0] = q.x; x[u][1] = q.y; x[u][2] = q.z; x[u][3] = q.w;
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) x[u][m] = 4 * g + m < np ? payload_word(src, nbytes, w + m) : 0;
        }
    }
}

template <int G, int CT>
__device__ __forceinline__ void slice_store(const LLArgs& a, int n, size_t w0, int np, int u0, uint32_t epoch,
                                            bool pk32, const uint32_t (&x)[8][4]) {
    const int items = n * G;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int it = threadIdx.x + (u0 + u) * CT;
        const int k = it / G, g = (it + 32 * k) % G;
        if (it >= items || 4 * g >= np) continue;
        uint64_t* dst = a.pkts[k] + w0 + 4 * g;
        if (4 * g + 4 <= np) {
            const uint64_t p0 = make_packet(x[u][0], epoch), p1 = make_packet(x[u][1], epoch);
            const uint64_t p2 = make_packet(x[u][2], epoch), p3 = make_packet(x[u][3], epoch);
            if (pk32) {
                st_packets4(dst, p0, p1, p2, p3);
            } else {
                st_packets2(dst, p0, p1);
                st_packets2(dst + 2, p2, p3);
            }
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (4 * g + m < np) st_packet(dst + m, make_packet(x[u][m], epoch));
        }
    }
}

template <int DT, int NR, int WB, int PPT>
__global__ void __launch_bounds__(kSliceThreads)
slice_kernel(const LLArgs a, int n_rt, size_t count, size_t nbytes, size_t slices, uint32_t host_epoch,
             uint64_t* ctrl, uint64_t max_spins, int32_t* status, bool in16, bool out16, bool pk32) {
    constexpr int CT = kSliceThreads;
    constexpr int SP = PPT * CT;
    constexpr int G = SP / 4;
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR > 0 ? (NR < 8 ? NR : 8) : 8;
    pdl_wait();
    const int n = ranks<NR>(n_rt);
    const size_t npk = (nbytes + 3) / 4;
    // The first window of input loads is issued before the epoch is known,
    // so those loads and the epoch counter's atomic are in flight together.
    uint32_t x[8][4];
    {
        const size_t w0 = static_cast<size_t>(blockIdx.x) * SP;
        slice_load<G, CT>(a, n, nbytes, in16, w0, static_cast<int>(min(static_cast<size_t>(SP), npk - w0)), 0, x);
    }
    __shared__ uint32_t s_epoch;
    if (threadIdx.x == 0) s_epoch = ctrl != nullptr ? take_ticket(ctrl) : host_epoch;
    __syncthreads();
    const uint32_t epoch = s_epoch;
    for (size_t b = blockIdx.x; b < slices; b += gridDim.x) {
        const size_t w0 = b * SP;
        const int np = static_cast<int>(min(static_cast<size_t>(SP), npk - w0));

        // A. send
        for (int u0 = 0; u0 * CT < n * G; u0 += 8) {
            if (b != blockIdx.x || u0 != 0) slice_load<G, CT>(a, n, nbytes, in16, w0, np, u0, x);
            slice_store<G, CT>(a, n, w0, np, u0, epoch, pk32, x);
        }

        // B. poll and reduce
        const int t0 = PPT * threadIdx.x;
        const int mn = min(PPT, np - t0);
        const size_t w = w0 + t0;
        float acc[PPT][EP];
        if (mn > 0) {
#pragma unroll 1
            for (int k0 = 0; k0 < n; k0 += WIN) {
                uint64_t pk[WIN][PPT];
#pragma unroll
                for (int k = 0; k < WIN; ++k) {
                    if (NR == 0 && k0 + k >= n) break;
                    const uint64_t* row = a.pkts[k0 + k] + w;
                    if (PPT == 4 && mn >= 4) {
                        ld_packets2(row, pk[k][0], pk[k][PPT > 1 ? 1 : 0]);
                        ld_packets2(row + 2, pk[k][PPT > 2 ? 2 : 0], pk[k][PPT > 3 ? 3 : 0]);
                    } else {
#pragma unroll
                        for (int m = 0; m < PPT; ++m) pk[k][m] = m < mn ? ld_packet(row + m) : 0;
                    }
                }
                unsigned ns = 32;
                for (uint64_t spin = 0;; ++spin) {
                    bool ready = true;
#pragma unroll
                    for (int k = 0; k < WIN; ++k) {
                        if (NR == 0 && k0 + k >= n) break;
#pragma unroll
                        for (int m = 0; m < PPT; ++m) ready = ready && (m >= mn || packet_flag(pk[k][m]) == epoch);
                    }
                    if (ready) break;
                    if (spin >= max_spins) {
                        atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
                        return;
                    }
                    if (spin >= kSpinPolls) {
                        if (ld_status_word(status) != 0) return;
                        __nanosleep(ns);
                        if (ns < kMaxSleepNs) ns *= 2;
                    }
#pragma unroll
                    for (int k = 0; k < WIN; ++k) {
                        if (NR == 0 && k0 + k >= n) break;
#pragma unroll
                        for (int m = 0; m < PPT; ++m)
                            if (m < mn && packet_flag(pk[k][m]) != epoch) pk[k][m] = ld_packet(a.pkts[k0 + k] + w + m);
                    }
                }
#pragma unroll
                for (int k = 0; k < WIN; ++k) {
                    if (NR == 0 && k0 + k >= n) break;
#pragma unroll
                    for (int m = 0; m < PPT; ++m) {
                        float xv[EP];
                        widen_word<DT>(packet_payload(pk[k][m]), xv);
#pragma unroll
                        for (int e = 0; e < EP; ++e) acc[m][e] = (k0 + k == 0) ? xv[e] : __fadd_rn(acc[m][e], xv[e]);
                    }
                }
            }

            // C. write-back
            if constexpr (WB == kDirect) {
                if (out16 && mn >= PPT && 4 * (w + PPT) <= nbytes) {
                    if constexpr (PPT == 4) {
                        const uint4 y = make_uint4(narrow_word<DT>(acc[0]), narrow_word<DT>(acc[PPT > 1 ? 1 : 0]),
                                                   narrow_word<DT>(acc[PPT > 2 ? 2 : 0]),
                                                   narrow_word<DT>(acc[PPT > 3 ? 3 : 0]));
                        for (int j = 0; j < n; ++j) st_stream(static_cast<uint4*>(a.data.out[j]) + w / 4, y);
                    } else {
                        const uint32_t y = narrow_word<DT>(acc[0]);
                        for (int j = 0; j < n; ++j) st_stream_word(static_cast<uint32_t*>(a.data.out[j]) + w, y);
                    }
                } else {
                    for (int m = 0; m < PPT && m < mn; ++m)
#pragma unroll
                        for (int e = 0; e < EP; ++e) {
                            const size_t i = (w + m) * EP + e;
                            if (i < count)
                                for (int j = 0; j < n; ++j) store_elem<DT>(a.data.out[j], i, acc[m][e]);
                        }
                }
            } else {
                // Elements past the end are zero bits, as in the send's padding.
                for (int m = 0; m < PPT && m < mn; ++m) {
                    float xs[EP];
#pragma unroll
                    for (int e = 0; e < EP; ++e) xs[e] = ((w + m) * EP + e < count) ? acc[m][e] : 0.0f;
                    st_packet(a.res + w + m, make_packet(narrow_word<DT>(xs), epoch));
                }
            }
        }
        if constexpr (WB == kPacketsAll) {
            // Result packets of the thread one warp further on: each read once
            // and written to every output.
            const int tr = (threadIdx.x + 32) % CT;
            const int mr = min(PPT, np - PPT * tr);
            if (mr > 0) {
                uint64_t r[PPT];
                load_slot<PPT>(a.res, w0 + PPT * tr, mr, r);
                if (!finish_slot<DT, PPT>(a, count, nbytes, w0 + PPT * tr, mr, 0, n, epoch, max_spins, status, out16,
                                          r))
                    return;
            }
        } else if constexpr (WB == kPacketsOwn) {
            // Item (j, q): output rank j reads result group q (4 packets) of
            // the slice and writes output j; the items are spread over the
            // threads (rotated by a warp per output rank), the loads of up to
            // 8 items issued before their polls.
            const int ngr = (np + 3) / 4;
            const int items = n * ngr;
            for (int u0 = 0; u0 * CT < items; u0 += 8) {
                uint64_t r[8][4];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int it = threadIdx.x + (u0 + u) * CT;
                    const int j = it / ngr, q = (it + 32 * (j + 1)) % ngr;
                    if (it < items) load_slot<4>(a.res, w0 + 4 * q, min(4, np - 4 * q), r[u]);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int it = threadIdx.x + (u0 + u) * CT;
                    const int j = it / ngr, q = (it + 32 * (j + 1)) % ngr;
                    if (it < items && !finish_slot<DT, 4>(a, count, nbytes, w0 + 4 * q, min(4, np - 4 * q), j, j + 1,
                                                          epoch, max_spins, status, out16, r[u]))
                        return;
                }
            }
        }
    }
}

// Blocks of the sliced form: one per slice, at most kMaxSliceBlocks (then each
// block takes several slices in turn; a launch's tickets stay below 2^20).
constexpr size_t kMaxSliceBlocks = size_t(1) << 16;

template <int DT, int NR, int WB>
cudaError_t slice_launch(int nranks, const LLArgs& a, size_t count, uint32_t epoch, uint64_t* ctrl,
                         uint64_t max_spins, int32_t* status, bool in16, bool out16, cudaStream_t s) {
    constexpr int PPT = kSlicePackets;
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    const size_t slices = (npk + PPT * kSliceThreads - 1) / (PPT * kSliceThreads);
    const unsigned blocks = static_cast<unsigned>(std::min(slices, kMaxSliceBlocks));
    bool p32 = true;
    for (int r = 0; r < nranks; ++r) p32 = p32 && reinterpret_cast<uintptr_t>(a.pkts[r]) % 32 == 0;
    return launch_kernel(slice_kernel<DT, NR, WB, PPT>, dim3(blocks), dim3(kSliceThreads), s, a, nranks, count,
                         nbytes, slices, epoch, ctrl, max_spins, status, in16, out16, p32);
}

inline unsigned div_up(size_t a, size_t b) { return static_cast<unsigned>((a + b - 1) / b); }

template <int DT, int NR, int WB>
cudaError_t coop_dispatch(int nranks, const LLArgs& a, size_t count, uint32_t epoch, uint64_t* ctrl,
                          uint64_t max_spins, int32_t* status, bool in16, bool out16, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    // Packets per rank, a multiple of 4 so that result groups never straddle two chunks.
    const size_t chunk = ((npk + nranks - 1) / nranks + 3) / 4 * 4;
    // Blocks per rank: enough threads for the largest phase, capped so that
    // all nranks * gx blocks are co-resident (resident blocks per SM x SMs,
    // looked up once per device).
    constexpr int kMaxDev = 64;
    static std::atomic<int> resident[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    int blocks = resident[dev].load(std::memory_order_relaxed);
    if (blocks == 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, coop_kernel<DT, NR, WB>, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks = sms * per_sm;
        resident[dev].store(blocks, std::memory_order_relaxed);
    }
    // (The up to 4 packets after the last whole 16 input bytes go to threads
    // 0..3 of a rank's first block, so they need no block of their own: an
    // idle extra block cost 1.4 us per call at 8 x 4 KiB.)
    size_t want = std::max<size_t>(div_up(in16 ? nbytes / 16 : npk, kThreads), div_up(chunk, kThreads));
    if (WB == kPacketsOwn) want = std::max<size_t>(want, div_up((npk + 3) / 4, kThreads));
    const size_t cap = static_cast<size_t>(blocks) / nranks;
    if (cap == 0) return cudaErrorCooperativeLaunchTooLarge;
    const unsigned gx = static_cast<unsigned>(std::max<size_t>(1, std::min(want, cap)));
    if (static_cast<uint64_t>(gx) * nranks > (uint64_t(1) << kTicketBits)) return cudaErrorInvalidConfiguration;
    LLArgs args = a;
    int n_rt = nranks;
    size_t cnt = count, nb = nbytes, cq = chunk;
    bool p32 = true;
    for (int r = 0; r < nranks; ++r) p32 = p32 && reinterpret_cast<uintptr_t>(a.pkts[r]) % 32 == 0;
    uint32_t ep = epoch;
    uint64_t* ct = ctrl;
    uint64_t ms = max_spins;
    int32_t* st = status;
    bool i16 = in16, o16 = out16;
    // Cooperative (every block co-resident) and, like the other kernels,
    // programmatic stream serialization: the kernel waits for the previous
    // one with pdl_wait() before touching memory.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, nranks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, coop_kernel<DT, NR, WB>, args, n_rt, cnt, nb, cq, ep, ct, ms, st, i16, o16,
                              p32);
}

// The sliced form for direct and multi-destination write-backs up to their
// size limits, the cooperative form otherwise.
template <int DT, int NR, int WB>
cudaError_t ll_dispatch(int nranks, const LLArgs& a, size_t count, uint32_t epoch, uint64_t* ctrl,
                        uint64_t max_spins, int32_t* status, bool in16, bool out16, cudaStream_t s) {
    const size_t bytes = count * Elem<DT>::kSize;
    const size_t limit = WB == kDirect ? kSliceDirectMaxBytes : (WB == kPacketsAll ? kSliceMultiDestMaxBytes : kSliceOwnMaxBytes);
    if (bytes <= limit)
        return slice_launch<DT, NR, WB>(nranks, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    return coop_dispatch<DT, NR, WB>(nranks, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
}

template <int DT, int WB>
cudaError_t coop_ranks(int nranks, const LLArgs& a, size_t count, uint32_t epoch, uint64_t* ctrl,
                       uint64_t max_spins, int32_t* status, bool in16, bool out16, cudaStream_t s) {
    switch (nranks) {
    case 1: return ll_dispatch<DT, 1, WB>(1, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    case 2: return ll_dispatch<DT, 2, WB>(2, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    case 4: return ll_dispatch<DT, 4, WB>(4, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    case 8: return ll_dispatch<DT, 8, WB>(8, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    case 16: return ll_dispatch<DT, 16, WB>(16, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    case 32: return ll_dispatch<DT, 32, WB>(32, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    default:
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        return ll_dispatch<DT, 0, WB>(nranks, a, count, epoch, ctrl, max_spins, status, in16, out16, s);
    }
}

template <int WB>
cudaError_t coop_launch(sar_dtype dt, int nranks, const RankPtrs& data, void* const* pkts, void* res, size_t count,
                        uint32_t epoch, uint64_t* ctrl, uint64_t max_spins, int32_t* status, bool in16, bool out16,
                        cudaStream_t stream) {
    LLArgs a;
    a.data = data;
    for (int r = 0; r < SAR_MAX_RANKS; ++r) a.pkts[r] = r < nranks ? static_cast<uint64_t*>(pkts[r]) : nullptr;
    a.res = static_cast<uint64_t*>(res);
#define SAR_COOP(T) coop_ranks<T, WB>(nranks, a, count, epoch, ctrl, max_spins, status, in16, out16, stream)
    switch (dt) {
    case SAR_BF16: return SAR_COOP(SAR_BF16);
    case SAR_FP16: return SAR_COOP(SAR_FP16);
    case SAR_FP32: return SAR_COOP(SAR_FP32);
    case SAR_FP8_E4M3FN: return SAR_COOP(SAR_FP8_E4M3FN);
    case SAR_FP8_E4M3B15: return SAR_COOP(SAR_FP8_E4M3B15);
    }
#undef SAR_COOP
    return cudaErrorInvalidValue;
}

}  // namespace llc
}  // namespace sar
