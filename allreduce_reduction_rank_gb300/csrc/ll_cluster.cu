// ll_cluster.cu -- the LL all-pair allreduce through distributed shared
// memory: the simulated ranks of one slice of the data are the CTAs of one
// thread-block cluster.
//
// mscclpp commit history, the allreduce_allpair_packet fix: each rank sends
// its data as flag-checked LL packets into every peer's scratch, the peer
// polls the flags in its own scratch, reduces and writes the result back,
// all in the same thread block.  On one GB300 the peers of a slice are the N
// CTAs of a cluster (CTA rank r = simulated rank r), and a CTA's scratch is
// its shared memory, which the other CTAs of the cluster write directly
// (st.shared::cluster to a mapa-translated address):
//
//   clear  : every CTA clears its packet slots (N x CT 8-byte packets)
//            and arrives at a cluster barrier; it loads its input words and
//            waits at the barrier before its first store into another CTA,
//            so no slot is written before its owner has cleared it;
//   send   : CTA k turns its input words for the slice of every chunk r into
//            packets {payload, flag} and stores them into CTA r's slots
//            [k][0..CT) (16-byte stores of two packets, each packet a
//            single-copy-atomic 8-byte element);
//   reduce : thread t of CTA r polls slot [k][t] for every k until its flag is
//            set (bounded; a timeout is recorded in the status word), adds the
//            payloads in rank order 0..N-1 in binary32, rounds once and writes
//            the result word to all N outputs;
//   exit   : every CTA arrives at a second cluster barrier after its last
//            store into another CTA and waits there before it leaves, so no
//            CTA leaves while another may still write into its shared memory.
//
// The slots start every launch at zero ("never written"), so every launch
// uses the flag value 1: no epoch is carried between launches and a CUDA
// graph can replay the call as it is.  Packets never touch global memory:
// HBM traffic is N*S read plus N*S written, as for the rsag kernel.  Clusters
// hold at most 16 CTAs (8 portably), so N <= 16.
//
// Slice of cluster `team` in chunk r: packets [r*chunk + team*CT, +CT)
// of the rank's packet range (chunk = packets per rank chunk, a multiple of
// 4), cut at the end of the chunk and of the buffer.  Packet w holds bytes
// 4w..4w+3 of a rank's input, zero past its end, as in sar_ll_pack.
#include <atomic>

#include "ll_packets.cuh"
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace llk {

constexpr int kMaxClusterRanks = SAR_LL_CLUSTER_MAX_RANKS;
constexpr uint32_t kFlag = 1;             // flag of a written slot (cleared slots hold 0)
constexpr uint64_t kSpinPolls = 16;       // immediate re-reads before a poll backs off
constexpr unsigned kMaxSleepNs = 1024;

// The two halves of a cluster barrier.  Arrive publishes this CTA's earlier
// memory operations (release); wait returns once every CTA of the cluster has
// arrived and makes theirs visible (acquire).  Work placed between the halves
// hides the barrier's latency.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of `local` (a shared::cta address) in CTA `rank` of
// this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster2(uint32_t addr, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.cluster.shared::cluster.v2.u64 [%0], {%1, %2};" :: "r"(addr), "l"(a), "l"(b)
                 : "memory");
}
__device__ __forceinline__ void st_cluster1(uint32_t addr, uint64_t a) {
    asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(a) : "memory");
}
__device__ __forceinline__ uint64_t ld_slot(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t packet(uint32_t payload) {
    return static_cast<uint64_t>(payload) | (static_cast<uint64_t>(kFlag) << 32);
}


// CT: threads per CTA, also the packets per rank of a slice (one per
// reducing thread).
template <int DT, int NR, int CT>
__global__ void __launch_bounds__(CT)
cluster_kernel(const RankPtrs p, int n_rt, size_t count, size_t nbytes, size_t chunk, uint64_t max_spins,
               int32_t* status, bool in16, bool out16) {
    extern __shared__ __align__(16) uint64_t slots[];   // [sender k][CT]
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR > 0 ? NR : 16;
    const int n = ranks<NR>(n_rt);
    const uint32_t me = blockIdx.x % static_cast<uint32_t>(n);      // CTA rank in the cluster = simulated rank
    const size_t team = blockIdx.x / static_cast<uint32_t>(n);
    const size_t npk = (nbytes + 3) / 4;
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(slots));

    // clear: no global memory is touched yet, so this overlaps the previous
    // kernel's drain (programmatic launch).  The barrier's wait comes only
    // before the first store into another CTA's slots.
    for (int i = threadIdx.x; i < n * CT; i += CT) slots[i] = 0;
    cluster_arrive();
    pdl_wait();

    // send: 4 packets (one 16-byte input vector) per item; item v covers
    // destination r = v / (CT/4), packets 4*(v % (CT/4)) .. +3 of the
    // slice.  A thread loads all of its items, then waits for the cluster,
    // then stores them.
    const unsigned char* src = static_cast<const unsigned char*>(p.in[me]);
    constexpr int kGroups = CT / 4;
    constexpr int kItems = ((NR > 0 ? NR : kMaxClusterRanks) * kGroups + CT - 1) / CT;
    uint32_t x[kItems][4];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int v = threadIdx.x + u * CT;
        const int r = v / kGroups, g = v % kGroups;
        const size_t lo = static_cast<size_t>(r) * chunk;
        const size_t end = min(npk, lo + chunk);
        const size_t w = lo + team * CT + 4 * static_cast<size_t>(g);
        x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0;
        if (v >= n * kGroups || w >= end) continue;
        if (in16 && 4 * (w + 4) <= nbytes) {
            const uint4 q = ld_stream(reinterpret_cast<const uint4*>(src) + w / 4);
            x[u][0] = q.x; x[u][1] = q.y; x[u][2] = q.z; x[u][3] = q.w;
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) x[u][m] = w + m < end ? payload_word(src, nbytes, w + m) : 0;
        }
    }
    cluster_wait();
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int v = threadIdx.x + u * CT;
        const int r = v / kGroups, g = v % kGroups;
        const size_t lo = static_cast<size_t>(r) * chunk;
        const size_t end = min(npk, lo + chunk);
        const size_t w = lo + team * CT + 4 * static_cast<size_t>(g);
        if (v >= n * kGroups || w >= end) continue;
        const uint32_t dst = map_to_rank(base + static_cast<uint32_t>((me * CT + 4 * g) * 8), r);
        if (w + 4 <= end) {
            st_cluster2(dst, packet(x[u][0]), packet(x[u][1]));
            st_cluster2(dst + 16, packet(x[u][2]), packet(x[u][3]));
        } else {
            for (int m = 0; m < 4 && w + m < end; ++m) st_cluster1(dst + 8 * m, packet(x[u][m]));
        }
    }
    // Every packet of this CTA is stored; the matching wait comes at the exit.
    cluster_arrive();

    // reduce: thread t owns packet w of this CTA's chunk slice.
    const size_t lo = static_cast<size_t>(me) * chunk;
    const size_t end = min(npk, lo + chunk);
    const size_t w = lo + team * CT + threadIdx.x;
    if (w < end) {
        uint64_t pk[WIN];
        const uint32_t mine = base + static_cast<uint32_t>(threadIdx.x * 8);
#pragma unroll
        for (int k = 0; k < WIN; ++k)
            if (NR > 0 || k < n) pk[k] = ld_slot(mine + static_cast<uint32_t>(k * CT * 8));
        unsigned ns = 32;
        bool ok = true;
        for (uint64_t spin = 0;; ++spin) {
            bool ready = true;
#pragma unroll
            for (int k = 0; k < WIN; ++k)
                if (NR > 0 || k < n) ready = ready && static_cast<uint32_t>(pk[k] >> 32) == kFlag;
            if (ready) break;
            if (spin >= max_spins) {
                if (status != nullptr) atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
                ok = false;
                break;
            }
            if (spin >= kSpinPolls) {
                if (status != nullptr && ld_status_word(status) != 0) {
                    ok = false;
                    break;
                }
                __nanosleep(ns);
                if (ns < kMaxSleepNs) ns *= 2;
            }
#pragma unroll
            for (int k = 0; k < WIN; ++k)
                if ((NR > 0 || k < n) && static_cast<uint32_t>(pk[k] >> 32) != kFlag)
                    pk[k] = ld_slot(mine + static_cast<uint32_t>(k * CT * 8));
        }
        if (ok) {
            float acc[EP];
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (NR == 0 && k >= n) break;
                float x[EP];
                widen_word<DT>(static_cast<uint32_t>(pk[k]), x);
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[e] = k == 0 ? x[e] : __fadd_rn(acc[e], x[e]);
            }
            if (out16 && 4 * (w + 1) <= nbytes) {
                const uint32_t y = narrow_word<DT>(acc);
#pragma unroll
                for (int j = 0; j < WIN; ++j)
                    if (NR > 0 || j < n) st_stream_word(static_cast<uint32_t*>(p.out[j]) + w, y);
            } else {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const size_t i = w * EP + e;
                    if (i < count)
                        for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], i, acc[e]);
                }
            }
        }
    }
    // exit: every CTA of the cluster has finished writing into the others'
    // slots before any of them leaves.
    cluster_wait();
}

template <int DT, int NR, int CT>
cudaError_t cluster_launch(int nranks, const RankPtrs& p, size_t count, size_t nbytes, size_t chunk,
                           uint64_t max_spins, int32_t* status, bool in16, bool out16, cudaStream_t s) {
    const size_t teams = (chunk + CT - 1) / CT;
    if (teams * static_cast<size_t>(nranks) > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(nranks) * CT * 8;
    // Clusters above 8 CTAs are not portable: allowed explicitly, once per
    // device and kernel (only a successful call is remembered).
    if (nranks > 8) {
        constexpr int kMaxDev = 64;
        static std::atomic<bool> allowed[kMaxDev];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
        if (!allowed[dev].load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(cluster_kernel<DT, NR, CT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            allowed[dev].store(true, std::memory_order_release);
        }
    }
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(nranks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(teams * static_cast<size_t>(nranks)));
    cfg.blockDim = dim3(CT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cluster_kernel<DT, NR, CT>, p, nranks, count, nbytes, chunk, max_spins, status,
                              in16, out16);
}

// Slice size (= threads per CTA): the smallest of 64, 128 and 256 packets
// per rank that keeps the grid within 128 CTAs for 64 and within 512 CTAs for
// 128.  Smaller slices put more CTAs, on more SMs, to work on small calls;
// larger ones keep large calls within the clusters that fit at once.
// Measured (graph, 8 ranks fp32, us per call for CTAs of 64 / 128 / 256
// threads): 4 KiB 1.89 / 2.05 / 2.30, 16 KiB 1.96 / 2.08 / 2.55, 64 KiB
// 2.35 / 2.28 / 2.54, 256 KiB 4.60 / 3.91 / 4.34, 1 MiB 15.8 / 11.3 / 11.4;
// 16 ranks, 16 KiB 2.72 / 3.26 / 4.52, 64 KiB 4.45 / 4.36 / 4.74.
template <int DT, int NR>
cudaError_t cluster_dispatch(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status,
                             bool in16, bool out16, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    const size_t chunk = ((npk + nranks - 1) / nranks + 3) / 4 * 4;
    const size_t n = static_cast<size_t>(nranks);
    if ((chunk + 63) / 64 * n <= 128)
        return cluster_launch<DT, NR, 64>(nranks, p, count, nbytes, chunk, max_spins, status, in16, out16, s);
    if ((chunk + 127) / 128 * n <= 512)
        return cluster_launch<DT, NR, 128>(nranks, p, count, nbytes, chunk, max_spins, status, in16, out16, s);
    return cluster_launch<DT, NR, 256>(nranks, p, count, nbytes, chunk, max_spins, status, in16, out16, s);
}

template <int DT>
cudaError_t cluster_ranks(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status,
                          bool in16, bool out16, cudaStream_t s) {
    switch (nranks) {
    case 1: return cluster_dispatch<DT, 1>(1, p, count, max_spins, status, in16, out16, s);
    case 2: return cluster_dispatch<DT, 2>(2, p, count, max_spins, status, in16, out16, s);
    case 4: return cluster_dispatch<DT, 4>(4, p, count, max_spins, status, in16, out16, s);
    case 8: return cluster_dispatch<DT, 8>(8, p, count, max_spins, status, in16, out16, s);
    case 16: return cluster_dispatch<DT, 16>(16, p, count, max_spins, status, in16, out16, s);
    default:
        if (nranks < 1 || nranks > kMaxClusterRanks) return cudaErrorInvalidValue;
        return cluster_dispatch<DT, 0>(nranks, p, count, max_spins, status, in16, out16, s);
    }
}

}  // namespace llk

cudaError_t launch_ll_cluster(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                              int32_t* status, bool in16, bool out16, cudaStream_t stream) {
    switch (dt) {
    case SAR_BF16: return llk::cluster_ranks<SAR_BF16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP16: return llk::cluster_ranks<SAR_FP16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP32: return llk::cluster_ranks<SAR_FP32>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3FN:
        return llk::cluster_ranks<SAR_FP8_E4M3FN>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3B15:
        return llk::cluster_ranks<SAR_FP8_E4M3B15>(nranks, p, count, max_spins, status, in16, out16, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sar
