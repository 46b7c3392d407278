// Device building blocks shared by the sampling and filter kernels (sm_103a).
//
// Execution model: one thread-block cluster of C CTAs per row, rank 0 the leader.
// A row is cut into segments of 128 * 2^shift elements (128 = one float4 per lane of
// a warp); CTA c owns a contiguous range of them.  Every CTA streams its range from
// HBM exactly once (pass 1) and keeps each segment's maximum order key and mass; it
// sends its totals to every CTA, its segment masses into the leader's shared memory
// when a draw over the whole row may need them (distributed shared memory stores),
// and, when a top-k bound is needed, the top of its histogram of segment maxima into
// every CTA's (distributed shared memory atomics).  After one cluster barrier every
// CTA can derive the same top-k bound and gather its candidates.  Paths that need the
// whole cluster afterwards are driven by the leader through commands written into the
// other CTAs' shared memory (a candidate collection, a two-pivot reduction, a 7-pivot
// threshold-search pass, a masked write, exit), each bracketed by two cluster
// barriers; when little data is left the leader finishes alone.  The top-p filter
// runs symmetric histogram passes instead (renorm.cu).  Every CTA executes the same
// sequence of cluster barriers.
//
// Code size is kept small on purpose: the work after pass 1 runs once per CTA, from a
// cold instruction cache, on every SM at the same moment.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Everything on the path of a call is inlined: an out-of-line call saves and restores
// live registers through the stack, and with most of the SM's on-chip memory given to
// shared memory those accesses miss L1.  Only rarely taken fallbacks stay out of line.
#define FS_COLD __noinline__

namespace fsd {

constexpr int NT = 256;                 // threads per CTA
constexpr int NW = NT / 32;             // warps per CTA
constexpr int BLK = 128;                // elements per block (one float4 per lane)
constexpr int TB = 4;                   // blocks per trip (double-buffered in pass 1)
constexpr int MAX_SEG_SHIFT = 2;        // at most 4 blocks per segment (V <= 2^21)
constexpr int NS_TARGET = 4096;         // segments per row (longer rows use longer segments)
constexpr int CAP = 1024;               // compact-list capacity (leader)
constexpr int SBH = 2;                  // blocks per half of a warp's staging buffer
constexpr int HBINS = 2048;             // histogram bins of the top-k bound (key >> 21)
constexpr int R_MAX = 256;              // rejection rounds before a row is invalid
constexpr int MAX_CLUSTER = 16;         // CTAs per row (above 8: non-portable cluster sizes)
constexpr int REDW = 128;               // words of block-reduction scratch
constexpr uint64_t NO_LIMIT = uint64_t(1) << 32;  // an upper key bound that excludes nothing
constexpr unsigned FULL = 0xffffffffu;

// Commands from the leader to the other CTAs of the cluster.
static_assert(2 * HBINS <= NW * 2 * SBH * BLK, "both top-k histograms live in the staging buffers");
static_assert(HBINS <= 2 * CAP, "a CTA's own histogram counts live in the compact list (values, then indices)");

// A (token index, value) pair packed into one 64-bit register.
__device__ __forceinline__ unsigned long long pack_jx(int j, float x) {
    return (static_cast<unsigned long long>(static_cast<uint32_t>(j)) << 32) | __float_as_uint(x);
}
__device__ __forceinline__ int unpack_j(unsigned long long p) { return static_cast<int>(p >> 32); }
__device__ __forceinline__ float unpack_x(unsigned long long p) { return __uint_as_float(static_cast<uint32_t>(p)); }

enum : int { CMD_EXIT = 0, CMD_PIVOT2 = 1, CMD_SEARCH = 2, CMD_WRITE = 4, CMD_COLLECT = 5 };

// ------------------------------------------------------------------ geometry

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Smallest shift s with ceil(V / (BLK << s)) <= NS_TARGET.
__host__ __device__ inline int seg_shift_for(int V) {
    int s = 0;
    while (s < MAX_SEG_SHIFT && (V + (BLK << s) - 1) / (BLK << s) > NS_TARGET) ++s;
    return s;
}

// A command (written by the leader into every CTA's copy).
struct alignas(16) Ctl {
    int cmd;
    int ia, ib;            // PIVOT2: which mass arrays receive the per-segment masses
    int flag;              // WRITE: row valid
    float f[4];            // pivots / denominator
    uint32_t u[4];         // key pivots / threshold; u[3] = interval low (BISECT)
    uint32_t hi_lo, hi_hi; // BISECT: 64-bit interval high
    uint32_t pad[2];
};

// One CTA's partial results, in the leader's shared memory (one record per rank).
// Word i < 4 is f[i]; word 4 + i is u[i].
struct alignas(16) Part {
    float f[4];
    uint32_t u[12];
};

// The dynamic shared-memory carve-up for `ns` segments per row: a fixed header (the
// command, the parts, reduction scratch), five per-segment arrays of nsp words each,
// the compact list and the per-warp staging buffers.
struct Layout {
    static constexpr size_t CTL = 0;
    static constexpr size_t PART = align16(CTL + sizeof(Ctl));
    static constexpr size_t RED = align16(PART + MAX_CLUSTER * sizeof(Part));
    static constexpr size_t MISC = align16(RED + REDW * sizeof(int));
    static constexpr size_t ARR = align16(MISC + 32 * sizeof(int));
    size_t nsp;   // words per per-segment array (ns + 1, rounded up to 4)
    __host__ __device__ explicit Layout(int ns) : nsp((size_t(ns) + 4) & ~size_t(3)) {}
    __host__ __device__ size_t arr(int i) const { return ARR + size_t(i) * nsp * 4; }
    __host__ __device__ size_t lv() const { return arr(5); }
    __host__ __device__ size_t li() const { return lv() + size_t(CAP) * 4; }
    __host__ __device__ size_t stage() const { return li() + size_t(CAP) * 4; }
    __host__ __device__ size_t total() const { return stage() + size_t(NW) * 2 * SBH * BLK * 4; }
    // Top-p histograms (filter kernels only, after pass 1): two receive buffers of
    // TOPPW 64-bit words (HBINS bins and two totals) over the per-segment arrays from
    // arr(1) on (the masses and the live list, unused on that path), and a local one
    // in the staging buffers, or after the receive buffers when those reach into them.
    static constexpr size_t TOPPW = HBINS + 2;
    __host__ __device__ size_t topp_recv(int i) const { return arr(1) + size_t(i) * TOPPW * 8; }
    __host__ __device__ size_t topp_local() const {
        return topp_recv(2) <= stage() ? stage() : topp_recv(2);
    }
    __host__ __device__ size_t topp_total() const {
        const size_t end = topp_local() + TOPPW * 8;
        return end > total() ? end : total();
    }
};

extern __shared__ __align__(16) unsigned char smem_raw[];

// Views of the carve-up.  Holds only the segment count, so that it travels in a
// register: every pointer is recomputed from the shared-memory base.
struct Smem {
    int ns;
    __device__ explicit Smem(int ns_) : ns(ns_) {}
    template <typename T>
    __device__ __forceinline__ T* at(size_t off) const { return reinterpret_cast<T*>(smem_raw + off); }
    __device__ __forceinline__ Ctl* ctl() const { return at<Ctl>(Layout::CTL); }            // current command
    __device__ __forceinline__ Part* part() const { return at<Part>(Layout::PART); }        // [MAX_CLUSTER]
    __device__ __forceinline__ int* red() const { return at<int>(Layout::RED); }            // [REDW] scratch
    __device__ __forceinline__ float* cmass() const { return at<float>(Layout::MISC); }     // [MAX_CLUSTER]
    __device__ __forceinline__ int* ctr() const { return at<int>(Layout::MISC + 64); }      // pass-1 trip counter
    __device__ __forceinline__ int* bcast() const { return at<int>(Layout::MISC + 80); }    // [4] CTA broadcast
    __device__ __forceinline__ uint32_t* prm() const { return at<uint32_t>(Layout::MISC + 96); }  // [8] row parameters
    __device__ __forceinline__ uint32_t* segkey() const { return at<uint32_t>(Layout(ns).arr(0)); }
    __device__ __forceinline__ float* mass(int i) const { return at<float>(Layout(ns).arr(1 + i)); }  // i < 3
    __device__ __forceinline__ int* list() const { return at<int>(Layout(ns).arr(4)); }     // live segments
    __device__ __forceinline__ float* lv() const { return at<float>(Layout(ns).lv()); }     // [CAP] values
    __device__ __forceinline__ int* li() const { return at<int>(Layout(ns).li()); }         // [CAP] indices
    // [HBINS] aliases the staging buffers: written (by every CTA) and read before any staging
    __device__ __forceinline__ uint32_t* hist() const { return at<uint32_t>(Layout(ns).stage()); }
    __device__ __forceinline__ float* stage() const { return at<float>(Layout(ns).stage()); }
    __device__ __forceinline__ unsigned long long* topp_recv(int i) const {
        return at<unsigned long long>(Layout(ns).topp_recv(i));
    }
    __device__ __forceinline__ unsigned long long* topp_local() const {
        return at<unsigned long long>(Layout(ns).topp_local());
    }
};

// The row, its segmentation and this CTA's share.  Segment indices are row-wide.
struct Geom {
    int V;
    int shift;     // log2(blocks per segment)
    int ns;        // segments per row
    int nsc;       // segments per CTA (the last may own fewer)
    int s0, s1;    // this CTA's segments [s0, s1)
    __device__ Geom(int V_, int shift_, int ns_, int nsc_, int rank) : V(V_), shift(shift_), ns(ns_), nsc(nsc_) {
        s0 = min(ns, rank * nsc);
        s1 = min(ns, s0 + nsc);
    }
    __device__ int seg_it() const { return 1 << shift; }
    // First element of block `it` of segment `s`, as seen by `lane`.
    __device__ int base(int s, int it, int lane) const { return ((s << shift) + it) * BLK + lane * 4; }
    // The segment range of rank c.
    __device__ void range_of(int c, int& a, int& b) const {
        a = min(ns, c * nsc);
        b = min(ns, a + nsc);
    }
    // Rows of logits sampled through a softmax: every value read from the row after the
    // row maximum vm is known is turned into its weight w = exp((z - vm) / T) (vinv =
    // 1 / T), so that the rest of the path works on unnormalised probabilities.  For
    // rows of probabilities (soft = false) values are used as they are.
    bool soft = false;
    float vm = 0.f, vinv = 1.f;
    // Chain speculative verification: values are the residual max(x - y, 0) of the
    // row against this second row at the same index (null: the row itself).
    const float* qrow = nullptr;
    __device__ __forceinline__ float val(float x) const { return soft ? expf((x - vm) * vinv) : x; }
    __device__ __forceinline__ float4 val4(float4 v) const {
        return soft ? make_float4(val(v.x), val(v.y), val(v.z), val(v.w)) : v;
    }
    // The raw value past the row end that stands for weight 0.
    __device__ __forceinline__ float fill0() const { return soft ? __int_as_float(0xff800000) : 0.f; }
};

// ------------------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Hardware cluster barrier with release/acquire ordering of shared memory at cluster
// scope.  Every thread of every CTA of the cluster must reach it; it also acts as a
// CTA-wide barrier.  The split form (arrive ... wait) lets independent work run
// between the two halves.
__device__ __forceinline__ void cluster_arrive() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    __syncwarp();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Store a word into the leader's copy of a shared-memory location (a local store on
// the leader itself).
__device__ __forceinline__ void put_leader(void* local_addr, uint32_t v, bool leader) {
    if (leader) {
        *reinterpret_cast<uint32_t*>(local_addr) = v;
    } else {
        st_dsmem_u32(map_rank(smem_u32(local_addr), 0), v);
    }
}
// Add n to a counter in the leader's shared memory.
__device__ __forceinline__ void add_leader(uint32_t* local_addr, uint32_t n, bool leader) {
    if (leader) {
        atomicAdd(local_addr, n);
    } else {
        asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(map_rank(smem_u32(local_addr), 0)), "r"(n)
                     : "memory");
    }
}

// Programmatic dependent launch.  grid_dependency_wait() returns once every kernel
// this grid depends on (the previous kernel of the stream) has completed and its
// memory operations are visible; it must precede the first global-memory access.
// allow_dependents() lets the next kernel of the stream be scheduled on SMs this grid
// leaves free; that kernel still waits for this grid's completion before it reads.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ loads

// Elements [base, base+4) that straddle the row end, or of an unaligned row: element
// by element, `fill` past V.  Out of line: the cold path.
template <bool NC>
FS_COLD __device__ float4 load4_tail(const float* __restrict__ row, int V, int base, float fill) {
    float t[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) t[q] = (base + q < V) ? (NC ? __ldg(row + base + q) : row[base + q]) : fill;
    return make_float4(t[0], t[1], t[2], t[3]);
}

// Four consecutive elements [base, base+4) of a row.  VEC: the row start is 16-byte
// aligned and V % 4 == 0.  NC: read-only (non-coherent) path, used by the samplers,
// whose input is never written during the kernel; the filters may run in place and
// read coherently.
template <bool VEC, bool NC>
__device__ __forceinline__ float4 load4(const float* __restrict__ row, int V, int base, float fill) {
    if (VEC && base + 3 < V) {
        if (NC) {
            float4 v;
            asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(row + base));
            return v;
        }
        return *reinterpret_cast<const float4*>(row + base);
    }
    return load4_tail<NC>(row, V, base, fill);
}

__device__ __forceinline__ float q_at(const float4& v, int q) {
    return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// max(x - y, 0), keeping a NaN difference so that the row shows as bad.
__device__ __forceinline__ float residual_of(float x, float y) {
    const float d = x - y;
    return (d > 0.f || d != d) ? d : 0.f;
}

// The lane's four values of the row at `base` as the path sees them: the row's own
// values or, with a second row, their residual against it; then the weight transform
// of rows of logits.
template <bool VEC, bool NC>
__device__ __forceinline__ float4 row4(const float* __restrict__ row, const Geom& g, int base, float fill) {
    float4 v = load4<VEC, NC>(row, g.V, base, fill);
    if (g.qrow) {
        const float4 y = load4<VEC, NC>(g.qrow, g.V, base, 0.f);
        v = make_float4(residual_of(v.x, y.x), residual_of(v.y, y.y), residual_of(v.z, y.z), residual_of(v.w, y.w));
    }
    return g.val4(v);
}

// Asynchronous copies global -> shared (cp.async, completed per thread by
// cp.async.wait_group).  `bytes` < the copy size zero-fills the rest, and 0 reads
// nothing; the source address is then the row start, which is always valid.
__device__ __forceinline__ void cp_async16(float* dst, const float* src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float* dst, const float* src, int bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Ask the memory system to bring elements [e0, e1) of a row into L2 (bulk L2 prefetch,
// no destination, nothing to wait for), split over the lanes of one warp in pieces of
// whole 16-byte words.  The row start must be 16-byte aligned and e0 % 4 == 0; the
// last piece ends at e1 rounded down to a multiple of 4 (a partial word is left to the
// ordinary loads).  Warp-collective.
__device__ __forceinline__ void l2_prefetch_range(const float* row, int e0, int e1, int lane) {
    const int words = max(0, (e1 - e0) >> 2);       // 16-byte words
    const int per = (words + 31) / 32;
    const int w0 = min(words, lane * per);
    const int w1 = min(words, w0 + per);
    if (w1 > w0) {
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row + e0 + 4 * w0), "r"(uint32_t(w1 - w0) * 16u)
                     : "memory");
    }
}

// Stage the lane's four elements [base, base+4) of a row into dst[0..4); zeros past V.
// VEC: the row start is 16-byte aligned and V % 4 == 0, so base < V implies base + 4 <= V.
template <bool VEC>
__device__ __forceinline__ void stage4(float* dst, const float* __restrict__ row, int V, int base) {
    if (VEC) {
        const bool in = base < V;
        cp_async16(dst, in ? row + base : row, in ? 16 : 0);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = base + q < V;
            cp_async4(dst + q, in ? row + base + q : row, in ? 4 : 0);
        }
    }
}

// ------------------------------------------------------------------ warp / block helpers

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
    return v;  // bitwise identical in every lane: each level adds a commuted pair
}
__device__ __forceinline__ int warp_sum_i(int v) { return __reduce_add_sync(FULL, v); }
__device__ __forceinline__ uint32_t warp_max_u(uint32_t v) { return __reduce_max_sync(FULL, v); }
__device__ __forceinline__ uint32_t warp_min_u(uint32_t v) { return __reduce_min_sync(FULL, v); }
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}
__device__ __forceinline__ int warp_incl_scan_i(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// Contiguous range of [0, n) handled by warp w of NW.
__device__ __forceinline__ void warp_range(int n, int w, int& r0, int& r1) {
    const int per = (n + NW - 1) / NW;
    r0 = min(n, w * per);
    r1 = min(n, r0 + per);
}

// Sum of a[a0..a1) in a fixed order by one warp: lane-strided, then a tree.
// Identical in all lanes.
__device__ __forceinline__ float warp_ordered_sum(const float* a, int a0, int a1, int lane) {
    float acc = 0.f;
    for (int i = a0 + lane; i < a1; i += 32) acc += a[i];
    return warp_sum(acc);
}

// Block-wide sum of a per-warp value (each warp passes its warp-uniform value);
// fixed order, every thread gets the result.
__device__ __forceinline__ int block_sum_warp_values(int v, int* red, int warp, int lane) {
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int s = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += red[w];
    __syncthreads();
    return s;
}

// ------------------------------------------------------------------ keys

// Order key of a probability: its bit pattern when positive, 0 for +-0.  For
// non-negative floats the integer order of the pattern is the numeric order
// ([drill] section 3).
__device__ __forceinline__ uint32_t prob_key(float x) { return x > 0.f ? __float_as_uint(x) : 0u; }

// x * 2^sh rounded to the nearest integer (halves up), for x >= 0, computed from the
// bits of x (x = m * 2^(e - 150) with the implicit bit in m; subnormals have e = 1 and
// no implicit bit).  The caller keeps x * 2^sh below 2^63, so m << s fits.
__device__ __forceinline__ unsigned long long fixed_point(float x, int sh) {
    const uint32_t b = __float_as_uint(x);
    int e = int(b >> 23);
    unsigned long long m = b & 0x7fffffu;
    if (e) m |= 0x800000u; else e = 1;
    const int s = e - 150 + sh;
    if (s >= 0) return m << s;
    if (s < -25) return 0ull;  // below one half
    return (m + (1ull << (-s - 1))) >> (-s);
}

// Order-preserving key of a signed float ([drill] section 8: negative patterns sort
// backwards, so they are flipped; non-negative ones get the sign bit set).
__device__ __forceinline__ uint32_t logit_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The float whose order key (logit_key) is k.
__device__ __forceinline__ float from_logit_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct KeyProb {
    __device__ __forceinline__ uint32_t operator()(float x) const { return prob_key(x); }
};
struct KeyLogit {
    __device__ __forceinline__ uint32_t operator()(float x) const { return logit_key(x); }
};

// ------------------------------------------------------------------ Philox4x32-10

// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11:
// ten rounds of two 32x32->64 multiplies with a Weyl key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k.x += W0; k.y += W1; }
        const uint32_t lo0 = M0 * c.x, hi0 = __umulhi(M0, c.x);
        const uint32_t lo1 = M1 * c.z, hi1 = __umulhi(M1, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    }
    return c;
}

// Uniform of output row `b`, round `r`: 24 random bits, exact in float32, in [0, 1).
__device__ __forceinline__ float sampler_uniform(unsigned long long seed, unsigned long long offset, uint32_t b,
                                                 uint32_t r) {
    const uint4 ctr = make_uint4(r, b, uint32_t(offset), uint32_t(offset >> 32));
    const uint2 key = make_uint2(uint32_t(seed), uint32_t(seed >> 32));
    return float(philox4x32_10(ctr, key).x >> 8) * 0x1p-24f;
}

// This warp's contiguous share of the CTA's segments, read again from global memory
// (in practice L2, after pass 1) in chunks of TB blocks held in registers, the next
// chunk's loads in flight while the current one is processed.  Blocks of segments
// with live(sg) false are not read.  Then, in block order, body(sg, it, on, v, base):
// `it` the block's index inside segment sg, `on` = live(sg), v the lane's four values
// (zeros when not on or past V), base the index of v.x.  NC: read-only loads (the row
// is not written during the kernel).
template <bool VEC, bool NC, typename LIVE, typename BODY>
__device__ __forceinline__ void stream_warp(const float* __restrict__ row, Geom g, Smem sm, int warp, int lane,
                                            LIVE live, BODY body) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const int nblk = (r1 - r0) << g.shift;
    const int mask = g.seg_it() - 1;
    auto load_chunk = [&](int b0, float4* v) {
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int blk = b0 + j;
            const int sg = r0 + (blk >> g.shift);
            v[j] = (blk < nblk && live(sg)) ? row4<VEC, NC>(row, g, g.base(sg, blk & mask, lane), g.fill0())
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float4 A[TB], Bv[TB];
    load_chunk(0, A);
#pragma unroll 1
    for (int b0 = 0; b0 < nblk; b0 += TB) {
        load_chunk(b0 + TB, Bv);
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int blk = b0 + j;
            if (blk < nblk) {
                const int sg = r0 + (blk >> g.shift);
                body(sg, blk & mask, live(sg), A[j], g.base(sg, blk & mask, lane));
            }
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) A[j] = Bv[j];
    }
}

// Warp-collective inclusive prefix sum of 64-bit words.
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}
__device__ __forceinline__ uint32_t warp_incl_scan_t(uint32_t v, int lane) { return uint32_t(warp_incl_scan_i(int(v), lane)); }
__device__ __forceinline__ unsigned long long warp_incl_scan_t(unsigned long long v, int lane) {
    return warp_incl_scan_u64(v, lane);
}

// Warp-collective: scanning the bins h[top], h[top - 1], ... h[0] from the top down,
// the first bin at which the running count (or mass) reaches kk (-1 when it never
// does), and in `above` the sum of the bins scanned before it.  Lane l holds four
// consecutive bins of each window of 128.
template <typename T>
__device__ __forceinline__ int scan_bins_down(const T* h, int top, T kk, int lane, T& above) {
    T before = 0;
    above = 0;
#pragma unroll 1
    for (; top >= 0; top -= 128) {
        T c[4], own = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int bin = top - 4 * lane - q;
            c[q] = bin >= 0 ? h[bin] : T(0);
            own += c[q];
        }
        const T incl = warp_incl_scan_t(own, lane);
        const T total = __shfl_sync(FULL, incl, 31);
        if (before + total >= kk) {
            const T excl = before + incl - own;
            const int l = __ffs(__ballot_sync(FULL, excl < kk && excl + own >= kk)) - 1;
            T cum = excl;
            int q = 0;  // the first of the lane's bins where the running sum reaches kk
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                cum += c[t];
                if (cum < kk) q = t + 1;
            }
            T ab = excl;
#pragma unroll
            for (int t = 0; t < 4; ++t) ab += t < q ? c[t] : T(0);
            above = __shfl_sync(FULL, ab, l);
            return __shfl_sync(FULL, top - 4 * lane - q, l);
        }
        before += total;
    }
    return -1;
}

// ------------------------------------------------------------------ pass 1

// One streaming pass over this CTA's segments, in trips of TB blocks (whole segments):
// warp w starts with trip w and then takes the next untaken trip from a shared counter
// (initialised to NW), so that warps finishing early take more; the next trip's loads
// are in flight while the current trip is reduced.  For every segment: the maximum order key and (PROB) the
// mass, into this CTA's table.  Per lane: the positive count, a bad-value flag (NaN
// or negative for probabilities, NaN for logits) and the largest key seen.  With
// `hist_shift` >= 0 every segment maximum is also counted into the CTA's local
// histogram (lv, cleared beforehand) at bin key >> hist_shift.  Touches no other CTA,
// so it may run before the cluster's first barrier completes.  `prologue` runs in
// every thread once the first trip's loads are issued (the block-wide set-up that the
// counter and the histogram need: it ends with a block barrier), so that set-up
// overlaps the first round trip to memory.
//
// SOFT (rows of logits sampled through a softmax, read once; PROB false): keys are
// logit keys, the positive count is the count of logits above -inf, and +inf is a bad
// value as well as NaN.  SOFT = 2 also keeps a segment's mass as sum exp((z - zmax) / T)
// relative to its own largest logit zmax (1/T = g.vinv), the running maximum of an
// online softmax; pass1_totals moves the masses to the CTA's maximum and the sampler to
// the row's.  SOFT = 1 keeps no masses (paths that draw only from gathered candidates).
struct NoPrologue {
    __device__ __forceinline__ void operator()() const {}
};
template <bool VEC, bool NC, bool PROB, int SOFT = 0, typename PRO = NoPrologue>
__device__ __forceinline__ void pass1(const float* __restrict__ row, Geom g, Smem sm, int hist_shift, int warp,
                                      int lane, int& pos, bool& bad, uint32_t& kmax, PRO prologue = PRO()) {
    const int spt = TB >> g.shift;  // segments per trip
    const int ntrip = (g.s1 - g.s0 + spt - 1) / spt;
    const int mask = g.seg_it() - 1;
    const float fill = PROB ? 0.f : __int_as_float(0xff800000);
    auto load_trip = [&](int t, float4* v) {
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int sg = g.s0 + t * spt + (j >> g.shift);
            v[j] = (t < ntrip && sg < g.s1)
                       ? row4<VEC, NC>(row, g, g.base(sg, j & mask, lane), g.soft ? g.fill0() : fill)
                       : make_float4(fill, fill, fill, fill);
        }
    };
    if (VEC && warp == 0)  // the CTA's whole share towards L2 at once; the loads below then mostly hit L2
        l2_prefetch_range(row, g.s0 * (BLK << g.shift), min(g.V, g.s1 * (BLK << g.shift)), lane);
    float4 A[TB], Bv[TB];
    int t = warp;  // the first NW trips are fixed; later ones are taken from the counter
    load_trip(t, A);
    prologue();  // block-wide set-up, while the first trip's loads are in flight
#pragma unroll 1
    while (t < ntrip) {
        int tn = 0;
        if (lane == 0) tn = atomicAdd(sm.ctr(), 1);
        tn = __shfl_sync(FULL, tn, 0);
        load_trip(tn, Bv);
        const int sg0 = g.s0 + t * spt;
        float s[TB];
        uint32_t km[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int sg = sg0 + (j >> g.shift);
            const int base = g.base(sg, j & mask, lane);
            uint32_t k = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(A[j], q);
                if (PROB) {
                    bad |= !(x >= 0.f);
                    k = max(k, prob_key(x));
                    pos += x > 0.f;
                } else {
                    const bool in = sg < g.s1 && base + q < g.V;
                    bad |= isnan(x);
                    if (SOFT) {
                        bad |= in && x == __int_as_float(0x7f800000);
                        pos += in && x > __int_as_float(0xff800000);
                    }
                    k = max(k, in ? logit_key(x) : 0u);
                }
            }
            km[j] = __reduce_max_sync(FULL, k);
            kmax = max(kmax, km[j]);
            s[j] = PROB ? (A[j].x + A[j].y) + (A[j].z + A[j].w) : 0.f;
        }
        if (SOFT == 2) {  // weights relative to each block's largest logit, all blocks at once
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                // a block of -inf or padding has no finite maximum: +inf makes its weights 0
                const float zb = km[j] > 0x007fffffu ? from_logit_key(km[j]) : __int_as_float(0x7f800000);
                float e = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) e += expf((q_at(A[j], q) - zb) * g.vinv);
                s[j] = e;
            }
        }
        if (PROB || SOFT == 2) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TB; ++j) s[j] += __shfl_xor_sync(FULL, s[j], m);
        }
        // Lane l stores segment sg0 + l, its blocks combined in order.
        const int sg = sg0 + lane;
        if (lane < spt && sg < g.s1) {
            float ss = 0.f;
            uint32_t kk = 0;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const bool mine = (j >> g.shift) == lane;
                ss += mine ? s[j] : 0.f;
                kk = mine ? max(kk, km[j]) : kk;
            }
            if (SOFT == 2 && g.shift > 0) {  // blocks of one segment: each to the segment's largest logit
                ss = 0.f;
                const float zs = from_logit_key(kk);
#pragma unroll
                for (int j = 0; j < TB; ++j)
                    if ((j >> g.shift) == lane && km[j] > 0x007fffffu)
                        ss += s[j] * expf((from_logit_key(km[j]) - zs) * g.vinv);
            }
            sm.segkey()[sg] = kk;
            if (PROB || SOFT == 2) sm.mass(0)[sg] = ss;
            if (hist_shift >= 0)  // this CTA's histogram counts, in lv
                atomicAdd(reinterpret_cast<uint32_t*>(sm.lv()) + min(uint32_t(HBINS - 1), kk >> hist_shift), 1u);
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) A[j] = Bv[j];
        t = tn;
    }
}

// Store a 16-byte word into rank r's copy of a shared-memory location.
__device__ __forceinline__ void st_rank_v4(void* local_addr, uint4 v, uint32_t r, uint32_t self) {
    if (r == self) {
        *reinterpret_cast<uint4*>(local_addr) = v;
    } else {
        asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(map_rank(smem_u32(local_addr), r)),
                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
    }
}

// After pass 1 and the cluster barrier that follows it, every CTA: with `publish`, its
// segments' masses into the leader's mass table (for draws over the whole row); its
// totals into part[rank] of every CTA (f[0] ordered mass of its segments, u[0]
// positive count, u[1] bad flag, u[2] maximum key); and, if `hist_shift` >= 0, the
// CTA's counts of its segment maxima (key >> hist_shift, made by pass 1 in lv) into the
// histogram of every CTA of the cluster, each of which cleared its own (and its lv)
// before that barrier.  With `hist_k` > 0 only the CTA's bins from its largest down to
// the one where its own count reaches hist_k are added: the cluster's count reaches
// hist_k at or above the highest such bin of any CTA, and every bin from there up is
// exact, so the top-k bound is the same.  The CTA's first segment is a multiple of 4,
// so the table moves in 16-byte words.  With `online` (pass 1 SOFT = 2) the segment masses are first moved
// from each segment's largest logit to the CTA's (times exp((zmax - zcta) / T)), so
// the table and f[0] are relative to the CTA's maximum logit, u[2].  Block-collective.
__device__ __forceinline__ void pass1_totals(Geom g, Smem sm, bool leader, int rank, int C, int pos, bool bad,
                                             uint32_t kmax, int hist_shift, bool prob, bool publish, int warp,
                                             int lane, int tid, bool online = false, int hist_k = 0) {
    __syncthreads();  // the table and the local histogram counts written by pass 1
    if (online) {
        if (lane == 0) sm.red()[warp] = int(kmax);  // kmax is the same in every lane of a warp
        __syncthreads();
        uint32_t mk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) mk = max(mk, uint32_t(sm.red()[w]));
        if (mk > 0x007fffffu) {  // a logit above -inf
            const float zc = from_logit_key(mk);
#pragma unroll 1
            for (int i = g.s0 + tid; i < g.s1; i += NT) {
                const uint32_t kk = sm.segkey()[i];
                sm.mass(0)[i] = kk > 0x007fffffu ? sm.mass(0)[i] * expf((from_logit_key(kk) - zc) * g.vinv) : 0.f;
            }
        }
        __syncthreads();
    }
    const uint32_t* loc = reinterpret_cast<const uint32_t*>(sm.lv());
    if (publish && !leader) {
#pragma unroll 1
        for (int i = g.s0 + 4 * tid; i < g.s1; i += 4 * NT) {
            const int nv = min(4, g.s1 - i);
            if (nv == 4) {
                st_rank_v4(&sm.mass(0)[i], *reinterpret_cast<const uint4*>(&sm.mass(0)[i]), 0, 1);
            } else {  // the row's last, partial word: never past this CTA's range
#pragma unroll 1
                for (int q = 0; q < nv; ++q) put_leader(&sm.mass(0)[i + q], __float_as_uint(sm.mass(0)[i + q]), false);
            }
        }
    }
    // Per warp: counts, flags, maximum and the ordered mass of a fixed share of segments.
    float ms = 0.f;
    if (prob) {
        int r0, r1;
        warp_range(g.s1 - g.s0, warp, r0, r1);
        ms = warp_ordered_sum(sm.mass(0), g.s0 + r0, g.s0 + r1, lane);
    }
    pos = warp_sum_i(pos);
    const int b = __any_sync(FULL, bad) ? 1 : 0;
    float* rf = reinterpret_cast<float*>(sm.red());
    if (lane == 0) {
        sm.red()[warp] = pos;
        sm.red()[NW + warp] = b;
        sm.red()[2 * NW + warp] = int(kmax);
        rf[3 * NW + warp] = ms;
    }
    __syncthreads();
    if (hist_shift >= 0) {  // every non-empty bin (of the top ones) added once into each CTA's histogram
        int top = HBINS - 1, lowest = 0;
        if (hist_k > 0) {
            if (warp == 0) {
                uint32_t mk = 0;
#pragma unroll
                for (int w = 0; w < NW; ++w) mk = max(mk, uint32_t(sm.red()[2 * NW + w]));
                const int tb = int(min(uint32_t(HBINS - 1), mk >> hist_shift));
                uint32_t ab;
                const int br = scan_bins_down<uint32_t>(loc, tb, uint32_t(hist_k), lane, ab);
                if (lane == 0) {
                    sm.bcast()[0] = tb;
                    sm.bcast()[1] = max(br, 0);
                }
            }
            __syncthreads();
            top = sm.bcast()[0];
            lowest = sm.bcast()[1];
        }
#pragma unroll 1
        for (int bin = lowest + tid; bin <= top; bin += NT) {
            const uint32_t n = loc[bin];
            if (n) {
                uint32_t* h = &sm.hist()[bin];
#pragma unroll 1
                for (int r = 0; r < C; ++r) {
                    if (r == rank) {
                        atomicAdd(h, n);
                    } else {
                        asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(map_rank(smem_u32(h), uint32_t(r))),
                                     "r"(n)
                                     : "memory");
                    }
                }
            }
        }
    }
    if (tid < C) {
        int p = 0, nb = 0;
        uint32_t mk = 0;
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            p += sm.red()[w];
            nb |= sm.red()[NW + w];
            mk = max(mk, uint32_t(sm.red()[2 * NW + w]));
            m += rf[3 * NW + w];
        }
        st_rank_v4(&sm.part()[rank].u[0], make_uint4(uint32_t(p), uint32_t(nb), mk, 0u), uint32_t(tid), uint32_t(rank));
        st_rank_v4(&sm.part()[rank].f[0], make_uint4(__float_as_uint(m), 0u, 0u, 0u), uint32_t(tid), uint32_t(rank));
    }
}

// The rejection round's fused reduction ([blog] dual pivot) over this CTA's segments
// whose maximum exceeds p1: per segment the mass above p1 and above p2 (local and in
// the leader's mass[ia] / mass[ib]; zero for skipped segments); the CTA's ordered
// sums and counts into the leader's part[rank] (f[0], f[1], u[0], u[1]).
// Block-collective.
template <bool VEC>
__device__ __forceinline__ void pivot_pass(const float* __restrict__ row, Geom g, Smem sm, bool leader,
                                       int rank, float p1, float p2, int ia, int ib, int warp, int lane, int tid) {
    const uint32_t kp1 = prob_key(p1);
    const int last = g.seg_it() - 1;
    int c1 = 0, c2 = 0;
    float sa = 0.f, sb = 0.f;
    stream_warp<VEC, true>(
        row, g, sm, warp, lane, [&](int sg) { return sm.segkey()[sg] > kp1; },
        [&](int sg, int it, bool on, const float4& v, int) {
            float a = 0.f, b = 0.f;
            if (on) {
                float w1[4], w2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x = q_at(v, q);
                    w1[q] = x > p1 ? x : 0.f;
                    w2[q] = x > p2 ? x : 0.f;
                    c1 += x > p1;
                    c2 += x > p2;
                }
                a = warp_sum((w1[0] + w1[1]) + (w1[2] + w1[3]));
                b = warp_sum((w2[0] + w2[1]) + (w2[2] + w2[3]));
            }
            sa = it ? sa + a : a;
            sb = it ? sb + b : b;
            if (it == last && lane == 0) {
                sm.mass(ia)[sg] = sa;
                sm.mass(ib)[sg] = sb;
                if (!leader) {
                    put_leader(&sm.mass(ia)[sg], __float_as_uint(sa), false);
                    put_leader(&sm.mass(ib)[sg], __float_as_uint(sb), false);
                }
            }
        });
    c1 = warp_sum_i(c1);
    c2 = warp_sum_i(c2);
    if (lane == 0) {
        sm.red()[warp] = c1;
        sm.red()[NW + warp] = c2;
    }
    __syncthreads();
    if (warp == 0) {
        const float t1 = warp_ordered_sum(sm.mass(ia), g.s0, g.s1, lane);
        const float t2 = warp_ordered_sum(sm.mass(ib), g.s0, g.s1, lane);
        if (lane == 0) {
            int n1 = 0, n2 = 0;
#pragma unroll 1
            for (int w = 0; w < NW; ++w) {
                n1 += sm.red()[w];
                n2 += sm.red()[NW + w];
            }
            uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part()[rank]);
            put_leader(dst + 0, __float_as_uint(t1), leader);
            put_leader(dst + 1, __float_as_uint(t2), leader);
            put_leader(dst + 4, uint32_t(n1), leader);
            put_leader(dst + 5, uint32_t(n2), leader);
        }
    }
    __syncthreads();
}

// Rows of logits sampled through a softmax, once the row maximum g.vm is known: this
// CTA's segment keys (logit keys of each segment's largest logit) become keys of the
// weights w = exp((z - vm) / T), raised by 4 units in the last place so that no weight
// of the segment exceeds its key whatever the last-place error of expf (within 2
// units; (z - vm) / T is correctly rounded, hence non-decreasing in z).
// Block-collective; the caller synchronises before the keys are read.
__device__ __forceinline__ uint32_t soft_weight_key(const Geom& g, uint32_t lk) {
    return lk > 0x007fffffu ? prob_key(expf((from_logit_key(lk) - g.vm) * g.vinv)) : 0u;
}
__device__ __forceinline__ void soft_segment_keys(const Geom& g, Smem sm, int tid) {
#pragma unroll 1
    for (int i = g.s0 + tid; i < g.s1; i += NT) {
        const uint32_t w = soft_weight_key(g, sm.segkey()[i]);
        sm.segkey()[i] = w == 0u ? 0u : min(w + 4u, 0x7f7fffffu);
    }
}
// The weight key of a lower bound L on logit keys, lowered by 8 units in the last
// place (at least 1): every weight whose logit is at least L, and the k-th largest
// weight when L is at most the k-th largest logit, lie at or above it.
__device__ __forceinline__ uint32_t soft_bound(const Geom& g, uint32_t L) {
    const uint32_t w = soft_weight_key(g, L);
    return w > 9u ? w - 8u : 1u;
}

// ------------------------------------------------------------------ candidate lists

// Every element with thr <= key < thr_hi of the segments [a, b), in index order:
// out(p, value, index) for p = 0, 1, ...  Returns the exact count (the same in every
// thread).  Each warp lists the segments of its contiguous share of [a, b) whose
// maximum key is >= thr (into list[], inside its share); after one block barrier the
// live blocks, in index order, are dealt round-robin to the warps, CB at a time, so
// that every warp stages at most CB / NW of them at once (cp.async, into its part of
// the staging area; a crowded share no longer serialises its warp); the blocks' counts
// meet in red[] and a second barrier turns them into output offsets.  Block-collective;
// red[0, NW + CB) is used, and the caller has synchronised the block since its own
// last use of red.
template <bool VEC, typename KEYF, typename OUT>
__device__ __forceinline__ int collect_range(const float* __restrict__ row, Geom g, Smem sm, int a, int b,
                                             uint32_t thr, uint64_t thr_hi, KEYF keyf, int warp, int lane,
                                             OUT out) {
    constexpr int PW = 2 * SBH;  // blocks per warp in flight: its staging buffer
    constexpr int CB = NW * PW;  // blocks per batch (one count per lane of a warp)
    static_assert(CB == 32 && NW + CB <= REDW, "a batch's counts fit one warp and the scratch");
    int r0, r1;
    warp_range(b - a, warp, r0, r1);
    r0 += a;
    r1 += a;
    // This warp's live segments, in order, into list[r0 ..).
    int nl = 0;
#pragma unroll 1
    for (int b0 = r0; b0 < r1; b0 += 32) {
        const int i = b0 + lane;
        const bool live = i < r1 && sm.segkey()[i] >= thr;
        const unsigned bal = __ballot_sync(FULL, live);
        if (live) sm.list()[r0 + nl + __popc(bal & ((1u << lane) - 1u))] = i;
        nl += __popc(bal);
    }
    if (lane == 0) sm.red()[warp] = nl;
    __syncthreads();
    // Lane w < NW: warp w's live count, the inclusive prefix over warps, and its share's start.
    const int wn = lane < NW ? sm.red()[lane] : 0;
    const int wincl = warp_incl_scan_i(wn, lane);
    int ws0, ws1;
    warp_range(b - a, lane < NW ? lane : 0, ws0, ws1);
    const int nblk = __shfl_sync(FULL, wincl, NW - 1) << g.shift;
    const int mask = g.seg_it() - 1;
    // The element base of live block j (in index order) for this lane.
    auto block_base = [&](int j) {
        const int s = j >> g.shift;  // its ordinal among the live segments
        const int w = __popc(__ballot_sync(FULL, lane < NW && wincl <= s));
        const int first = __shfl_sync(FULL, wincl - wn, w);
        const int start = __shfl_sync(FULL, ws0, w) + a;
        return g.base(sm.list()[start + s - first], j & mask, lane);
    };
    auto keep = [&](float x, int base, int q) {
        const uint32_t key = keyf(g.val(x));
        return key >= thr && uint64_t(key) < thr_hi && base + q < g.V;
    };
    float* st = sm.stage() + warp * (PW * BLK) + lane * 4;
    int total = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < nblk; c0 += CB) {
        if (c0) __syncthreads();  // every warp has read the previous batch's counts
        int bs[PW];
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const int j = c0 + warp + NW * i;
            bs[i] = j < nblk ? block_base(j) : 0;
            if (j < nblk) stage4<VEC>(st + i * BLK, row, g.V, bs[i]);
        }
        cp_async_commit();
        cp_async_wait<0>();  // each lane reads back only the words it staged
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const int j = c0 + warp + NW * i;
            if (j < nblk) {
                int k = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) k += keep(st[i * BLK + q], bs[i], q);
                k = warp_sum_i(k);
                if (lane == 0) sm.red()[NW + (j - c0)] = k;
            }
        }
        __syncthreads();
        // Lane l: the count of the batch's block l and the inclusive prefix.
        const int bc = c0 + lane < nblk ? sm.red()[NW + lane] : 0;
        const int bincl = warp_incl_scan_i(bc, lane);
#pragma unroll 1
        for (int i = 0; i < PW; ++i) {
            const int jl = warp + NW * i;
            if (c0 + jl < nblk) {
                int p = total + __shfl_sync(FULL, bincl - bc, jl);
                int k = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) k += keep(st[i * BLK + q], bs[i], q);
                const int incl = warp_incl_scan_i(k, lane);
                p += incl - k;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (keep(st[i * BLK + q], bs[i], q)) out(p++, g.val(st[i * BLK + q]), bs[i] + q);
            }
        }
        total += __shfl_sync(FULL, bincl, 31);
    }
    return total;
}

// Every CTA: collect its own elements with thr <= key < thr_hi, in index order, into entries
// [base, base + cap) of the leader's list, or with `to_all` of every CTA's list; with
// `bcast`, the exact count goes to part[rank].u[4] of every CTA of the cluster, so that
// after the next cluster barrier each CTA can tell whether all regions fit and where
// each rank's candidates start.  Block-collective.
template <bool VEC, typename KEYF>
__device__ __forceinline__ void collect_own(const float* __restrict__ row, Geom g, Smem sm, bool leader, int rank,
                                            int C, int base, int cap, uint32_t thr, uint64_t thr_hi, KEYF keyf,
                                            bool to_all, bool bcast, int warp, int lane, int tid) {
    const int n = collect_range<VEC>(row, g, sm, g.s0, g.s1, thr, thr_hi, keyf, warp, lane, [&](int p, float x,
                                                                                                  int ix) {
        if (p < cap) {
            if (to_all) {
#pragma unroll 1
                for (int r = 0; r < C; ++r) {
                    if (r == rank) {
                        sm.lv()[base + p] = x;
                        sm.li()[base + p] = ix;
                    } else {
                        st_dsmem_u32(map_rank(smem_u32(&sm.lv()[base + p]), uint32_t(r)), __float_as_uint(x));
                        st_dsmem_u32(map_rank(smem_u32(&sm.li()[base + p]), uint32_t(r)), uint32_t(ix));
                    }
                }
            } else {
                put_leader(&sm.lv()[base + p], __float_as_uint(x), leader);
                put_leader(&sm.li()[base + p], uint32_t(ix), leader);
            }
        }
    });
    if (bcast && tid < C) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part()[rank]) + 8;
        if (tid == rank) {
            *dst = uint32_t(n);
        } else {
            st_dsmem_u32(map_rank(smem_u32(dst), uint32_t(tid)), uint32_t(n));
        }
    }
}

// After the barrier that follows collect_own: whether every rank's candidates fit in
// its region, and their total.  Any CTA (each holds every count); warp-parallel, every
// lane of every warp gets the result.
__device__ __forceinline__ bool regions_fit(Smem sm, int C, int rc) {
    const int lane = threadIdx.x & 31;
    return __all_sync(FULL, lane >= C || int(sm.part()[lane].u[4]) <= rc);
}
__device__ __forceinline__ int regions_total(Smem sm, int C) {
    const int lane = threadIdx.x & 31;
    return warp_sum_i(lane < C ? int(sm.part()[lane].u[4]) : 0);
}

// The cluster's totals from the parts written by pass1_totals (lane c reads part c).
struct Totals {
    int npos;
    bool any_bad;
    float M;
    uint32_t maxkey;
};
__device__ __forceinline__ Totals cluster_totals(Smem sm, int C) {
    const int lane = threadIdx.x & 31;
    const bool in = lane < C;
    const Part& p = sm.part()[in ? lane : 0];
    Totals t;
    t.npos = warp_sum_i(in ? int(p.u[0]) : 0);
    t.any_bad = __any_sync(FULL, in && p.u[1] != 0u);
    t.M = warp_sum(in ? p.f[0] : 0.f);
    t.maxkey = warp_max_u(in ? p.u[2] : 0u);
    return t;
}

// Start of rank r's candidates in the list: r * rc in region layout, or the count of
// the lower ranks when the list is contiguous.  Warp-parallel (lane r reads count r).
__device__ __forceinline__ int exact_base(Smem sm, int rank) {
    const int lane = threadIdx.x & 31;
    return warp_sum_i(lane < rank ? int(sm.part()[lane].u[4]) : 0);
}

// After a region collection and the cluster barrier that follows it, on every CTA
// alike: 0 when every region fit (the list stays in regions of CAP / C); 1 when a
// region overflowed but the total fits, after every CTA collected again at exact
// offsets and the cluster synchronised (the list is contiguous, in index order); -1
// when more than CAP elements qualify.  Block-collective on every CTA.
template <bool VEC, typename KEYF>
__device__ __forceinline__ int settle_list(const float* __restrict__ row, Geom g, Smem sm, bool leader, int rank,
                                           int C, uint32_t thr, uint64_t thr_hi, KEYF keyf, bool to_all, int warp,
                                           int lane, int tid) {
    if (regions_fit(sm, C, CAP / C)) return 0;
    if (regions_total(sm, C) > CAP) return -1;
    const int base = exact_base(sm, rank);
    collect_own<VEC>(row, g, sm, leader, rank, C, base, CAP - base, thr, thr_hi, keyf, to_all, false, warp, lane,
                     tid);
    cluster_sync();
    return 1;
}

// The candidate regions of all ranks, concatenated in rank order at the front of
// lv/li, by one warp.  Returns the total (the caller checked that every region fit).
// Regions only move towards the front and each chunk of 32 is read before it is
// written, so no entry is overwritten before it has been read.
__device__ __forceinline__ int join_regions_warp(Smem sm, int C, int rc, int lane) {
    int dst = 0;
#pragma unroll 1
    for (int c = 0; c < C; ++c) {
        const int n = int(sm.part()[c].u[4]);
        const int src = c * rc;
        if (src != dst) {
#pragma unroll 1
            for (int e0 = 0; e0 < n; e0 += 32) {
                const int e = e0 + lane;
                float v = 0.f;
                int ix = 0;
                if (e < n) {
                    v = sm.lv()[src + e];
                    ix = sm.li()[src + e];
                }
                __syncwarp();
                if (e < n) {
                    sm.lv()[dst + e] = v;
                    sm.li()[dst + e] = ix;
                }
                __syncwarp();
            }
        }
        dst += n;
    }
    return dst;
}

// A candidate list of at most SMALL entries held by one warp in registers, lane-major:
// entry e = SR * lane + r in slot r (x[r], i[r]); in[r] marks entries below n.
constexpr int SR = 4;              // slots per lane
constexpr int SMALL = 32 * SR;
struct Small {
    float x[SR];
    int i[SR];
    bool in[SR];
    int n;
};

// Gather the candidate list (counts in part[r].u[4], in rank order; rank r's entries
// start at r * rc, or with `exact` right after the lower ranks') n <= SMALL.
// Warp-collective.
__device__ __forceinline__ Small small_gather(Smem sm, int C, int rc, bool exact, int lane) {
    // Exclusive prefix of the region counts, region r's offset in lane r.
    const int cnt = lane < C ? int(sm.part()[lane].u[4]) : 0;
    const int off = warp_incl_scan_i(cnt, lane) - cnt;
    Small s;
    s.n = __shfl_sync(FULL, off + cnt, 31);
    int rr[SR], oo[SR];
#pragma unroll
    for (int r = 0; r < SR; ++r) {
        rr[r] = 0;
        oo[r] = 0;
    }
#pragma unroll 1
    for (int c = 0; c < C; ++c) {
        const int o = __shfl_sync(FULL, off, c);
        const int m = __shfl_sync(FULL, cnt, c);
#pragma unroll
        for (int r = 0; r < SR; ++r) {
            if (m > 0 && o <= SR * lane + r) {
                rr[r] = c;
                oo[r] = o;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < SR; ++r) {
        const int e = SR * lane + r;
        s.in[r] = e < s.n;
        const int a = exact ? e : rr[r] * rc + (e - oo[r]);
        s.x[r] = s.in[r] ? sm.lv()[a] : 0.f;
        s.i[r] = s.in[r] ? sm.li()[a] : 0;
    }
    return s;
}

// The k-th largest order key of a small list (0 if it has fewer than k entries): the
// largest key v with #{keys >= v} >= k.  When few entries lie below it (n - k < 32),
// the smallest keys are taken away one distinct value at a time (a warp minimum per
// step) until fewer than k would remain; otherwise every entry counts how many
// entries are at least as large (every entry visits every other through shuffles).
// Warp-collective.  Entries of the list have non-zero keys.
template <typename KEYF>
__device__ __forceinline__ uint32_t small_kth(const Small& s, int k, KEYF keyf) {
    if (s.n < k) return 0u;
    uint32_t key[SR];
#pragma unroll
    for (int r = 0; r < SR; ++r) key[r] = s.in[r] ? keyf(s.x[r]) : 0u;
    const int drop = s.n - k;  // entries strictly below the answer, at most
    if (drop < 32) {
        uint32_t floor_ = 0u;  // keys <= floor_ are taken away
        int gone = 0;
#pragma unroll 1
        for (int it = 0; it <= drop; ++it) {
            uint32_t m = 0xffffffffu;
#pragma unroll
            for (int r = 0; r < SR; ++r) m = (s.in[r] && key[r] > floor_) ? min(m, key[r]) : m;
            m = warp_min_u(m);
            int c = 0;
#pragma unroll
            for (int r = 0; r < SR; ++r) c += (s.in[r] && key[r] == m);
            c = warp_sum_i(c);
            if (gone + c > drop) return m;  // fewer than k would remain above m
            gone += c;
            floor_ = m;
        }
        return floor_;  // not reached: the loop ends by the return above
    }
    int ge[SR];
#pragma unroll
    for (int r = 0; r < SR; ++r) ge[r] = 0;
    const int lanes = (s.n + SR - 1) / SR;  // lanes holding entries
#pragma unroll 1
    for (int l = 0; l < lanes; ++l) {
#pragma unroll
        for (int r2 = 0; r2 < SR; ++r2) {
            const uint32_t a = __shfl_sync(FULL, key[r2], l);
#pragma unroll
            for (int r = 0; r < SR; ++r) ge[r] += int(a >= key[r]);
        }
    }
    uint32_t best = 0u;
#pragma unroll
    for (int r = 0; r < SR; ++r) best = max(best, s.in[r] && ge[r] >= k ? key[r] : 0u);
    return warp_max_u(best);
}

// In-place, order-preserving filter of lv/li[0..n) to key >= t by one warp.
// Returns the new length (warp-uniform).
template <typename KEYF>
__device__ __forceinline__ int filter_list_warp(Smem sm, int n, uint32_t t, KEYF keyf, int lane) {
    int w = 0;
#pragma unroll 1
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const bool keep = i < n && keyf(sm.lv()[i]) >= t;
        const float xv = keep ? sm.lv()[i] : 0.f;
        const int xi = keep ? sm.li()[i] : 0;
        const unsigned bal = __ballot_sync(FULL, keep);
        const int pos = w + __popc(bal & ((1u << lane) - 1u));
        __syncwarp();
        if (keep) {
            sm.lv()[pos] = xv;
            sm.li()[pos] = xi;
        }
        __syncwarp();
        w += __popc(bal);
    }
    return w;
}

// Block- and cluster-collective (every CTA of the cluster calls it with the same row,
// k and histogram): a lower bound L <= t_k of the row's k-th largest order key from
// the histogram of the segment maxima (key >> 21) that pass 1 left in every CTA.
// Scanning from the bin of the row maximum `maxkey` down, the bin B in which the
// count reaches k holds the k-th largest segment maximum, and its lower edge is at
// most that value.  The k-th largest of any subset of the row (here, the segment
// maxima) is at most the row's own k-th largest, so B's edge is <= t_k, and every
// segment holding an element >= t_k has its maximum >= the edge.
//
// A bin spans a quarter of a binade, which for logits of a few units is several units
// wide: when more than SMALL segment maxima are at or above B's edge, the bound is
// refined inside B.  Each CTA counts its own segment maxima that fall in B by the key
// bits 20..10 (in lv), adds the non-empty counts into every CTA's second histogram
// (which is zero since the kernel cleared it before its first cluster barrier), and
// after one cluster barrier every CTA scans B's 2048 sub-bins for the remaining k
// minus the count above B: the same argument, at 1/2048 of the width.  lv is free:
// no CTA writes candidates before the barrier.  Returns 0 when fewer than k
// segments exist.
__device__ __forceinline__ uint32_t hist_bound(Smem sm, Geom g, int rank, int C, int k, uint32_t maxkey, int warp,
                                               int lane, int tid) {
    if (g.ns < k) return 0;
    const uint32_t* h = sm.hist();
    if (warp == 0) {
        uint32_t above;
        const int B = scan_bins_down<uint32_t>(h, int(maxkey >> 21), uint32_t(k), lane, above);
        if (lane == 0) {
            sm.bcast()[0] = max(B, 0);
            sm.bcast()[1] = int(above);
            sm.bcast()[2] = B >= 0 ? int(above + h[B]) : 0;
        }
    }
    __syncthreads();
    const uint32_t B = uint32_t(sm.bcast()[0]);
    const int above = sm.bcast()[1];
    const int at = sm.bcast()[2];
    if (at <= SMALL) return B << 21;
    // ---- refinement inside bin B
    uint32_t* loc = reinterpret_cast<uint32_t*>(sm.lv());
    uint32_t* h2 = sm.hist() + HBINS;
#pragma unroll
    for (int q = 0; q < HBINS / NT; ++q) loc[q * NT + tid] = 0u;
    __syncthreads();
#pragma unroll 1
    for (int i = g.s0 + tid; i < g.s1; i += NT) {
        const uint32_t key = sm.segkey()[i];
        if ((key >> 21) == B) atomicAdd(&loc[(key >> 10) & (HBINS - 1)], 1u);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < HBINS / NT; ++q) {
        const int bin = q * NT + tid;
        const uint32_t n = loc[bin];
        if (n) {
#pragma unroll 1
            for (int r = 0; r < C; ++r) {
                if (r == rank) {
                    atomicAdd(&h2[bin], n);
                } else {
                    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(map_rank(smem_u32(&h2[bin]), uint32_t(r))),
                                 "r"(n)
                                 : "memory");
                }
            }
        }
    }
    cluster_sync();  // every CTA's counts are in every second histogram
    if (warp == 0) {
        uint32_t above2;
        const int top = (maxkey >> 21) == B ? int((maxkey >> 10) & (HBINS - 1)) : HBINS - 1;
        const int b2 = scan_bins_down<uint32_t>(h2, top, uint32_t(k - above), lane, above2);
        if (lane == 0) sm.bcast()[3] = max(b2, 0);
    }
    __syncthreads();
    return (B << 21) | (uint32_t(sm.bcast()[3]) << 10);
}

// Block-collective: the k-th largest order key of the list lv[0, n) (0 when n < k), by
// a most-significant-digit radix select over 8-bit digits: each round counts the
// keys that match the digits chosen so far into 256 counters (the histogram area of
// shared memory), warp 0 finds the digit at which the count from the top reaches
// the remaining rank, and the keys above that digit leave the rank.  The result is
// the same key as the warp's bit-by-bit search: the largest t with
// #{key >= t} >= k, which is a key of the list.
template <typename KEYF>
__device__ __forceinline__ uint32_t kth_key_cta(Smem sm, int n, int k, KEYF keyf, int warp, int lane, int tid) {
    static_assert(NT == 256, "one counter per thread");
    if (n < k) return 0u;
    uint32_t* h = sm.hist();
    uint32_t prefix = 0, pmask = 0, kk = uint32_t(k);
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        h[tid] = 0u;
        __syncthreads();
#pragma unroll 1
        for (int i = tid; i < n; i += NT) {
            const uint32_t key = keyf(sm.lv()[i]);
            if ((key & pmask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], own = 0;  // lane l: digits 255 - 8l down to 248 - 8l
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = h[255 - 8 * lane - q];
                own += c[q];
            }
            const uint32_t incl = uint32_t(warp_incl_scan_i(int(own), lane));
            const uint32_t excl = incl - own;
            const int l = __ffs(__ballot_sync(FULL, excl < kk && incl >= kk)) - 1;
            uint32_t cum = excl, ab = excl;
            int q = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                cum += c[t];
                if (cum < kk) q = t + 1;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) ab += t < q ? c[t] : 0u;
            const int d = __shfl_sync(FULL, 255 - 8 * lane - q, l);
            ab = __shfl_sync(FULL, ab, l);
            if (lane == 0) {
                sm.bcast()[0] = d;
                sm.bcast()[1] = int(ab);
            }
        }
        __syncthreads();
        prefix |= uint32_t(sm.bcast()[0]) << shift;
        pmask |= 255u << shift;
        kk -= uint32_t(sm.bcast()[1]);
    }
    return prefix;
}

// ------------------------------------------------------------------ draws

// Inverse-transform locate inside one segment, warp-collective ([blog] inverse
// transform sampling; implementation details: a parallel float prefix sum need not be
// monotone, so the result is always forced onto an eligible token).  Eligible: x >
// low.  `t` is the target measured from the segment start.  Returns the first
// eligible element whose running sum exceeds t, else the segment's last eligible
// element (-1 if none), packed with its value.
template <bool VEC, bool NC>
__device__ __forceinline__ unsigned long long locate_in_segment(const float* __restrict__ row, Geom g, int s, float low,
                                                            float t, int lane) {
    float run = 0.f;
    int last_j = -1;
    float last_x = 0.f;
#pragma unroll 1
    for (int it = 0; it < g.seg_it(); ++it) {
        const int base = g.base(s, it, lane);
        const float4 v = row4<VEC, NC>(row, g, base, g.fill0());
        float w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = q_at(v, q);
            w[q] = x > low ? x : 0.f;
        }
        const float lsum = (w[0] + w[1]) + (w[2] + w[3]);
        const bool any = (w[0] > 0.f) | (w[1] > 0.f) | (w[2] > 0.f) | (w[3] > 0.f);
        const float incl = warp_incl_scan(lsum, lane);
        const unsigned hit = __ballot_sync(FULL, any && (run + incl > t));
        const unsigned elig = __ballot_sync(FULL, any);
        if (elig) {
            const int l = 31 - __clz(elig);
            int lq = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (w[q] > 0.f) lq = q;
            const int lq_l = __shfl_sync(FULL, lq, l);
            last_j = __shfl_sync(FULL, base, l) + lq_l;
            last_x = __shfl_sync(FULL, q_at(v, lq), l);
        }
        if (hit) {
            const int l = __ffs(hit) - 1;
            int pq = -1, lastq = 0;
            float acc = run + (incl - lsum);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (w[q] > 0.f) {
                    acc += w[q];
                    lastq = q;
                    if (pq < 0 && acc > t) pq = q;
                }
            }
            if (pq < 0) pq = lastq;
            return pack_jx(__shfl_sync(FULL, base + pq, l), __shfl_sync(FULL, q_at(v, pq), l));
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    return pack_jx(last_j, last_x);
}

// One block of the guarded locate ([blog] implementation details): the lane's four
// values v are elements base .. base + 3 of the row (the lanes in index order) and are
// eligible when above low.  Returns true, with the pick packed in jx, when the running
// sum passes t inside the block; otherwise adds the block's eligible mass to run and
// remembers its last eligible element.  Warp-collective.
__device__ __forceinline__ bool locate_step(const float4& v, int base, float low, float t, float& run, int& last_j,
                                            float& last_x, unsigned long long& jx, int lane) {
    float w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float x = q_at(v, q);
        w[q] = x > low ? x : 0.f;
    }
    const float lsum = (w[0] + w[1]) + (w[2] + w[3]);
    const bool any = (w[0] > 0.f) | (w[1] > 0.f) | (w[2] > 0.f) | (w[3] > 0.f);
    const float incl = warp_incl_scan(lsum, lane);
    const unsigned hit = __ballot_sync(FULL, any && (run + incl > t));
    const unsigned elig = __ballot_sync(FULL, any);
    if (elig) {
        const int l = 31 - __clz(elig);
        int lq = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (w[q] > 0.f) lq = q;
        const int lq_l = __shfl_sync(FULL, lq, l);
        last_j = __shfl_sync(FULL, base, l) + lq_l;
        last_x = __shfl_sync(FULL, q_at(v, lq), l);
    }
    if (hit) {
        const int l = __ffs(hit) - 1;
        int pq = -1, lastq = 0;
        float acc = run + (incl - lsum);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (w[q] > 0.f) {
                acc += w[q];
                lastq = q;
                if (pq < 0 && acc > t) pq = q;
            }
        }
        if (pq < 0) pq = lastq;
        jx = pack_jx(__shfl_sync(FULL, base + pq, l), __shfl_sync(FULL, q_at(v, pq), l));
        return true;
    }
    run += __shfl_sync(FULL, incl, 31);
    return false;
}

// The guarded locate over the TB blocks of unit un of the row (a unit of the scan):
// the first element above low whose running sum passes t, else the last element above
// low (-1 if none), packed with its value.  Every block's load is issued before the
// first is scanned.  Warp-collective.
template <bool VEC>
__device__ __forceinline__ unsigned long long locate_in_unit(const float* __restrict__ row, int V, int un, float low,
                                                             float t, int lane) {
    float4 v[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j) v[j] = load4<VEC, true>(row, V, (un * TB + j) * BLK + lane * 4, 0.f);
    float run = 0.f;
    int last_j = -1;
    float last_x = 0.f;
    unsigned long long jx = 0ull;
#pragma unroll
    for (int j = 0; j < TB; ++j)
        if (locate_step(v[j], (un * TB + j) * BLK + lane * 4, low, t, run, last_j, last_x, jx, lane)) return jx;
    return pack_jx(last_j, last_x);
}

// First segment in [a, b) whose running mass over mass[] exceeds t; if none, the last
// segment with positive mass (-1 if none).  Packed with the mass before it.
// Warp-collective.
__device__ __forceinline__ unsigned long long locate_segment(const float* mass, int a, int b, float t, int lane) {
    float run = 0.f;
    int last = -1;
    float last_before = 0.f;
#pragma unroll 1
    for (int base = a; base < b; base += 32) {
        const float m = (base + lane < b) ? mass[base + lane] : 0.f;
        const float incl = warp_incl_scan(m, lane);
        const unsigned hit = __ballot_sync(FULL, m > 0.f && run + incl > t);
        const unsigned nz = __ballot_sync(FULL, m > 0.f);
        if (nz) {
            const int l = 31 - __clz(nz);
            last = base + l;
            last_before = run + __shfl_sync(FULL, incl - m, l);
        }
        if (hit) {
            const int l = __ffs(hit) - 1;
            return pack_jx(base + l, run + __shfl_sync(FULL, incl - m, l));
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    return pack_jx(last, last_before);
}

// Locate inside a compact list lv[0..n) (index order), eligible x > low.  Warp-collective.
__device__ __forceinline__ int locate_in_list(const float* lv, int n, float low, float t, int lane) {
    float run = 0.f;
    int last = -1;
#pragma unroll 1
    for (int base = 0; base < n; base += 128) {
        float w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = base + lane * 4 + q;
            const float x = e < n ? lv[e] : 0.f;
            w[q] = x > low ? x : 0.f;
        }
        const float lsum = (w[0] + w[1]) + (w[2] + w[3]);
        const bool any = (w[0] > 0.f) | (w[1] > 0.f) | (w[2] > 0.f) | (w[3] > 0.f);
        const float incl = warp_incl_scan(lsum, lane);
        const unsigned hit = __ballot_sync(FULL, any && (run + incl > t));
        const unsigned elig = __ballot_sync(FULL, any);
        if (elig) {
            const int l = 31 - __clz(elig);
            int lq = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (w[q] > 0.f) lq = q;
            last = base + l * 4 + __shfl_sync(FULL, lq, l);
        }
        if (hit) {
            const int l = __ffs(hit) - 1;
            int pq = -1, lastq = 0;
            float acc = run + (incl - lsum);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (w[q] > 0.f) {
                    acc += w[q];
                    lastq = q;
                    if (pq < 0 && acc > t) pq = q;
                }
            }
            if (pq < 0) pq = lastq;
            return base + l * 4 + __shfl_sync(FULL, pq, l);
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    return last;
}

// Inverse-transform draw over the whole row while its tokens are spread over the
// cluster (warp-collective, leader): the owning CTA from the per-CTA masses cmass[]
// (the first CTA whose running mass passes the target), the segment inside its range from
// mass[cur], then the token inside the segment.  Returns the token (-1 if none) packed
// with its value.
template <bool VEC>
__device__ __forceinline__ unsigned long long draw_full(const float* __restrict__ row, Geom g, Smem sm, int C, int cur,
                                                   float low, float target, int lane) {
    float run = 0.f, before = 0.f, last_before = 0.f;
    int owner = -1, last = -1;
    for (int c = 0; c < C; ++c) {
        const float m = sm.cmass()[c];
        if (m > 0.f) {
            if (owner < 0 && run + m > target) {
                owner = c;
                before = run;
            }
            last = c;
            last_before = run;
        }
        run += m;
    }
    if (owner < 0) {
        owner = last;
        before = last_before;
    }
    if (owner < 0) return pack_jx(-1, 0.f);
    int a0, a1;
    g.range_of(owner, a0, a1);
    float t = target - before;
    const unsigned long long ls = locate_segment(sm.mass(cur), a0, a1, t, lane);
    const int s = unpack_j(ls);
    if (s < 0) return pack_jx(-1, 0.f);
    t = (t - unpack_x(ls) < 0.f) ? 0.f : t - unpack_x(ls);
    return locate_in_segment<VEC, true>(row, g, s, low, t, lane);
}

// ------------------------------------------------------------------ commands

// Leader: publish a command into every CTA's Ctl (thread r writes rank r's copy, four
// 16-byte stores), then the cluster barrier after which the peers read it.
// Block-collective on the leader.
__device__ __forceinline__ void send_command(Smem sm, const Ctl& c, int C, int tid) {
    static_assert(sizeof(Ctl) == 64, "Ctl is four 16-byte words");
    if (tid < C) {
        const uint4 w[4] = {
            make_uint4(uint32_t(c.cmd), uint32_t(c.ia), uint32_t(c.ib), uint32_t(c.flag)),
            make_uint4(__float_as_uint(c.f[0]), __float_as_uint(c.f[1]), __float_as_uint(c.f[2]),
                       __float_as_uint(c.f[3])),
            make_uint4(c.u[0], c.u[1], c.u[2], c.u[3]),
            make_uint4(c.hi_lo, c.hi_hi, 0u, 0u)};
        uint4* dst = reinterpret_cast<uint4*>(sm.ctl());
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (tid == 0) {
                dst[i] = w[i];
            } else {
                asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 map_rank(smem_u32(dst + i), uint32_t(tid))),
                             "r"(w[i].x), "r"(w[i].y), "r"(w[i].z), "r"(w[i].w)
                             : "memory");
            }
        }
    }
    cluster_sync();
}

// ------------------------------------------------------------------ threshold search

// Search for the threshold of a filter over the integer order keys ([drill] sections
// 2-4: a count or a mass that is monotone in the threshold, searched on the fp32 bit
// pattern so that it ends exactly on a value of the row): the largest t with
// crit(t) = count(key >= t) >= k, or mass(key >= t) >= target.  Invariant: crit(lo)
// holds, crit(hi) does not; the counts and masses of keys >= hi are known.  Each pass
// splits [lo, hi) at NP pivots and measures, for every pivot, the count and mass of the
// keys in [pivot, hi).  Once at most CAP keys lie in [lo, hi) they are gathered on chip
// and the search ends there.
constexpr int NP = 7;
constexpr int INT_BIG = 0x7fffffff;

struct Search {
    uint64_t lo, hi;
    float mass_lo;   // mass(key >= lo)
    float mass_hi;   // mass(key >= hi)
    int cnt_hi;      // count(key >= hi)
    int cnt_in;      // count(lo <= key < hi), INT_BIG if not known
};

// Pivot i (0 <= i < NP) of [lo, hi): evenly spread; when the interval is short, lo + 1,
// lo + 2, ... (those reaching hi are inert: nothing in [lo, hi) is >= hi).
__device__ __forceinline__ uint64_t search_pivot(uint64_t lo, uint64_t hi, int i) {
    const uint64_t d = hi - lo;
    return d > uint64_t(NP) ? lo + (d * uint64_t(i + 1)) / uint64_t(NP + 1) : min(lo + uint64_t(i + 1), hi);
}

// Per-thread accumulation of one element into the NP pivot sums (mass when MASS;
// counts always).
// Keys, bounds and pivots are 32-bit here: hi <= maxkey + 1 and a valid row's largest
// key is below 0xffffffff (that pattern is a NaN), so min(hi, 0xffffffff) loses nothing.
template <bool MASS>
__device__ __forceinline__ void search_add(uint32_t key, float x, uint32_t lo, uint32_t hi, const uint32_t* piv,
                                           float* m, int* c) {
    if (key < lo || key >= hi) return;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const bool ge = key >= piv[i];
        if (MASS) m[i] += ge ? x : 0.f;
        c[i] += ge;
    }
}
__device__ __forceinline__ uint32_t clamp32(uint64_t v) { return uint32_t(min(v, uint64_t(0xffffffffu))); }

// Block: the NP sums of every thread, reduced in a fixed order, into the 2 * NP words
// of dst (masses as float bits, then counts), written by thread 0 through `put`.
template <typename PUT>
__device__ __forceinline__ void search_reduce(Smem sm, float* m, int* c, int warp, int lane, int tid, PUT put) {
    float* rf = reinterpret_cast<float*>(sm.red());
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        m[i] = warp_sum(m[i]);
        c[i] = warp_sum_i(c[i]);
    }
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            rf[i * NW + warp] = m[i];
            sm.red()[(NP + i) * NW + warp] = c[i];
        }
    }
    __syncthreads();
    if (tid < 2 * NP) {
        uint32_t v;
        if (tid < NP) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) a += rf[tid * NW + w];
            v = __float_as_uint(a);
        } else {
            int a = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) a += sm.red()[tid * NW + w];
            v = uint32_t(a);
        }
        put(tid, v);
    }
    __syncthreads();
}
static_assert(2 * NP * NW <= REDW, "search sums fit the reduction scratch");

// One pass of the search over this CTA's segments whose maximum key is >= lo; the
// record (words 0..NP-1 masses (when MASS), NP..2NP-1 counts) goes to the leader's
// part[rank].  Block-collective.
template <bool VEC, bool NC, bool MASS, typename KEYF>
__device__ __forceinline__ void search_pass(const float* __restrict__ row, Geom g, Smem sm, bool leader, int rank,
                                            uint64_t lo, uint64_t hi, KEYF keyf, int warp, int lane, int tid) {
    uint32_t piv[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) piv[i] = clamp32(search_pivot(lo, hi, i));
    const uint32_t lo32 = uint32_t(lo), hi32 = clamp32(hi);
    float m[NP];
    int c[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        m[i] = 0.f;
        c[i] = 0;
    }
    stream_warp<VEC, NC>(
        row, g, sm, warp, lane, [&](int sg) { return sm.segkey()[sg] >= lo32; },
        [&](int, int, bool on, const float4& v, int base) {
            if (!on) return;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (base + q < g.V) search_add<MASS>(keyf(q_at(v, q)), q_at(v, q), lo32, hi32, piv, m, c);
            }
        });
    uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part()[rank]);
    search_reduce(sm, m, c, warp, lane, tid, [&](int w, uint32_t v) { put_leader(dst + w, v, leader); });
}

// Fold the sums of a pass (masses M[i], counts N[i] of keys in [pivot i, hi)) into
// the search state; the criterion is on the mass (CRIT_MASS) or on the count.
template <bool CRIT_MASS>
__device__ __forceinline__ void search_update(Search& st, const float* M, const int* N, int kcrit, float target) {
    int best = -1;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const bool ok = CRIT_MASS ? (st.mass_hi + M[i] >= target) : (st.cnt_hi + N[i] >= kcrit);
        if (ok) best = i;
    }
    const uint64_t lo = st.lo, hi = st.hi;
    const int nxt = best + 1;  // the pivot that becomes hi (NP: hi stays)
    int cnt_lo_in = st.cnt_in;  // count of [new lo, old hi)
    if (best >= 0) {
        st.lo = search_pivot(lo, hi, best);
        st.mass_lo = st.mass_hi + M[best];
        cnt_lo_in = N[best];
    }
    if (nxt < NP) {
        st.hi = search_pivot(lo, hi, nxt);
        st.mass_hi += M[nxt];
        st.cnt_hi += N[nxt];
        st.cnt_in = cnt_lo_in == INT_BIG ? INT_BIG : cnt_lo_in - N[nxt];
    } else {
        st.cnt_in = cnt_lo_in;
    }
}

// Leader, with the cluster: passes over the row until the interval is exact or holds
// at most CAP keys (at most 40 passes).  MASS: masses are measured (probabilities);
// CRIT_MASS: the criterion is on them.  Block-collective on the leader.
template <bool VEC, bool NC, bool CRIT_MASS, bool MASS, typename KEYF>
__device__ __forceinline__ void search_row(const float* __restrict__ row, Geom g, Smem sm, int C, Search& st,
                                           int kcrit, float target, KEYF keyf, int warp, int lane, int tid) {
#pragma unroll 1
    for (int iter = 0; iter < 40 && st.hi - st.lo > 1 && st.cnt_in > CAP; ++iter) {
        Ctl c{};
        c.cmd = CMD_SEARCH;
        c.flag = MASS ? 1 : 0;
        c.u[0] = uint32_t(st.lo);
        c.hi_lo = uint32_t(st.hi);
        c.hi_hi = uint32_t(st.hi >> 32);
        send_command(sm, c, C, tid);
        search_pass<VEC, NC, MASS>(row, g, sm, true, 0, st.lo, st.hi, keyf, warp, lane, tid);
        cluster_sync();  // every part is in
        float M[NP];
        int N[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const bool in = lane < C;
            const uint32_t* w = reinterpret_cast<const uint32_t*>(&sm.part()[in ? lane : 0]);
            M[i] = warp_sum(in ? __uint_as_float(w[i]) : 0.f);
            N[i] = warp_sum_i(in ? int(w[NP + i]) : 0);
        }
        search_update<CRIT_MASS>(st, M, N, kcrit, target);
        __syncthreads();  // the parts are read before the next pass writes them
    }
}

// The search over a list lv/li[0..n) that holds every key of [lo, hi) (and no other),
// block-collective, until the interval is exact.
template <bool CRIT_MASS, bool MASS, typename KEYF>
__device__ __forceinline__ void search_list(Smem sm, int n, Search& st, int kcrit, float target, KEYF keyf,
                                            int warp, int lane, int tid) {
#pragma unroll 1
    for (int iter = 0; iter < 40 && st.hi - st.lo > 1; ++iter) {
        uint32_t piv[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) piv[i] = clamp32(search_pivot(st.lo, st.hi, i));
        const uint32_t lo32 = uint32_t(st.lo), hi32 = clamp32(st.hi);
        float m[NP];
        int c[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            m[i] = 0.f;
            c[i] = 0;
        }
#pragma unroll 1
        for (int e = tid; e < n; e += NT) search_add<MASS>(keyf(sm.lv()[e]), sm.lv()[e], lo32, hi32, piv, m, c);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part()[0]);  // 2 * NP words (free once gathered)
        search_reduce(sm, m, c, warp, lane, tid, [&](int w, uint32_t v) { dst[w] = v; });
        float M[NP];
        int N[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            M[i] = __uint_as_float(dst[i]);
            N[i] = int(dst[NP + i]);
        }
        search_update<CRIT_MASS>(st, M, N, kcrit, target);
        __syncthreads();
    }
}

// Leader: every element with thr <= key < thr_hi, in index order, into lv/li[0..n), on the
// leader's command.  The whole cluster collects (each CTA its own segments, into its
// region of the leader's list; again at exact offsets if a region overflowed).
// Returns n, or -1 when more than CAP elements qualify (the peers then still wait for
// commands).  With `exit_if_fit` the peers have left whenever n >= 0.
//
// With `count_u` >= 0 the leader already holds each CTA's exact count of those
// elements, in part[r].u[count_u] (from the last reduction, with at most CAP in all):
// CTA r's base offset (the sum of the counts before it) goes into its bcast[2] with
// the command (ib = 1), so the CTAs write one contiguous list at once and nothing
// overflows or needs collecting again.
template <bool VEC, typename KEYF>
__device__ __forceinline__ int gather_leader(const float* __restrict__ row, Geom g, Smem sm, int C, uint32_t thr,
                                             uint64_t thr_hi, KEYF keyf, bool exit_if_fit, int warp, int lane,
                                             int tid, int count_u = -1) {
    const int rc = CAP / C;
    Ctl c{};
    c.cmd = CMD_COLLECT;
    c.flag = exit_if_fit ? 1 : 0;
    c.u[0] = thr;
    c.hi_lo = uint32_t(thr_hi);
    c.hi_hi = uint32_t(thr_hi >> 32);
    if (count_u >= 0) {
        c.ib = 1;
        if (tid < C) {  // thread r: rank r's base offset, into rank r's bcast[2]
            int base = 0;
#pragma unroll 1
            for (int r = 0; r < tid; ++r) base += int(sm.part()[r].u[count_u]);
            if (tid == 0) {
                sm.bcast()[2] = base;
            } else {
                st_dsmem_u32(map_rank(smem_u32(&sm.bcast()[2]), uint32_t(tid)), uint32_t(base));
            }
        }
        int total = 0;
#pragma unroll 1
        for (int r = 0; r < C; ++r) total += int(sm.part()[r].u[count_u]);
        send_command(sm, c, C, tid);  // its barrier also publishes the bases
        collect_own<VEC>(row, g, sm, true, 0, C, 0, CAP, thr, thr_hi, keyf, false, false, warp, lane, tid);
        cluster_sync();  // every CTA's elements are in place
        return total;
    }
    send_command(sm, c, C, tid);
    collect_own<VEC>(row, g, sm, true, 0, C, 0, rc, thr, thr_hi, keyf, false, true, warp, lane, tid);
    cluster_sync();  // every region and count is in
    const int mode = settle_list<VEC>(row, g, sm, true, 0, C, thr, thr_hi, keyf, false, warp, lane, tid);
    if (mode < 0) return -1;
    const int n = regions_total(sm, C);
    if (mode == 0) {
        if (warp == 0) join_regions_warp(sm, C, rc, lane);
        __syncthreads();
    }
    return n;
}

// Leader: the threshold of a count (k) or mass (target) criterion over the row, from
// the state `st` (crit(st.lo) holds), with the cluster: passes over the row, then the
// remaining keys gathered on chip.  Returns with st.hi = st.lo + 1 (st.lo the
// threshold, st.mass_lo its mass), unless more than 40 passes were needed.
template <bool VEC, bool NC, bool CRIT_MASS, bool MASS, typename KEYF>
__device__ __forceinline__ void threshold_search(const float* __restrict__ row, Geom g, Smem sm, int C, Search& st,
                                                 int kcrit, float target, KEYF keyf, int warp, int lane, int tid) {
    search_row<VEC, NC, CRIT_MASS, MASS>(row, g, sm, C, st, kcrit, target, keyf, warp, lane, tid);
    if (st.hi - st.lo <= 1 || st.cnt_in > CAP) return;
    const int n = gather_leader<VEC>(row, g, sm, C, uint32_t(st.lo), st.hi, keyf, false, warp, lane, tid);
    if (n < 0) return;
    search_list<CRIT_MASS, MASS>(sm, n, st, kcrit, target, keyf, warp, lane, tid);
}

// The starting state of a search over a whole row: [0, maxkey + 1), everything in it.
__device__ __forceinline__ Search search_start(uint32_t maxkey, float M, int V) {
    Search st;
    st.lo = 0;
    st.hi = uint64_t(maxkey) + 1;
    st.mass_lo = M;
    st.mass_hi = 0.f;
    st.cnt_hi = 0;
    st.cnt_in = V;
    return st;
}

}  // namespace fsd
