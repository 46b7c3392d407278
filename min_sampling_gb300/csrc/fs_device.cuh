// Device building blocks shared by the sampling and filter kernels (sm_103a).
//
// Execution model: one thread-block cluster per row.  A row is cut into segments of
// 128 * 2^shift elements (128 = one float4 per lane of a warp); the C CTAs of a
// cluster own contiguous ranges of segments.  Every CTA streams its range from HBM
// exactly once (pass 1) and keeps, per segment, the maximum order key and the mass
// above the current lower pivot in shared memory.  Later work (rejection rounds,
// threshold searches, the filter write) visits only segments whose maximum can
// matter, re-reading them through L2, and switches to a compact in-shared-memory
// list of surviving tokens as soon as it is small.  Cross-CTA reductions go through
// distributed shared memory (mapa + ld.shared::cluster) and hardware cluster
// barriers; every CTA of a cluster executes the same sequence of cluster barriers,
// because every branch around one depends only on cluster-wide reduced values.
//
// Code size matters as much as instruction count here: the per-row work after pass 1
// runs once per CTA, so it executes from a cold instruction cache.  Hot loops are
// written out explicitly; everything that runs once per phase is kept out of line.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define FS_NOINLINE __noinline__

namespace fsd {

constexpr int NT = 256;                 // threads per CTA
constexpr int NW = NT / 32;             // warps per CTA
constexpr int BLK = 128;                // elements per block (one float4 per lane)
constexpr int TRIP = 8;                 // blocks a warp keeps in flight per trip
constexpr int MAX_SEG_SHIFT = 2;        // at most 4 blocks per segment (V <= 2^21 needs 2)
constexpr int NS_TARGET = 4096;         // segments per row (larger rows use longer segments)
constexpr int CAP = 2048;               // compact-list capacity per CTA / per row
constexpr int R_MAX = 256;              // rejection rounds before a row is invalid
constexpr int MAX_CLUSTER = 8;
constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------ geometry

struct Slot {            // one cluster-exchange record (80 bytes)
    float f[8];
    uint32_t u[12];
};

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Smallest shift s with ceil(V / (BLK << s)) <= NS_TARGET.
__host__ __device__ inline int seg_shift_for(int V) {
    int s = 0;
    while (s < MAX_SEG_SHIFT && (V + (BLK << s) - 1) / (BLK << s) > NS_TARGET) ++s;
    return s;
}

// Byte offsets of the dynamic shared-memory carve-up for `nsc` segments per CTA.
struct Layout {
    size_t slot, gath, redf, redi, misc, segkey, mass0, mass1, mass2, off, lv, li, total;
    __host__ __device__ explicit Layout(int nsc) {
        size_t o = 0;
        slot = o;   o = align16(o + 2 * sizeof(Slot));
        gath = o;   o = align16(o + MAX_CLUSTER * sizeof(Slot));
        redf = o;   o = align16(o + NW * 4 * sizeof(float));
        redi = o;   o = align16(o + NW * 4 * sizeof(int));
        misc = o;   o = align16(o + 32 * sizeof(int));
        segkey = o; o = align16(o + size_t(nsc) * 4);
        mass0 = o;  o = align16(o + size_t(nsc) * 4);
        mass1 = o;  o = align16(o + size_t(nsc) * 4);
        mass2 = o;  o = align16(o + size_t(nsc) * 4);
        off = o;    o = align16(o + size_t(nsc + 1) * 4);
        lv = o;     o = align16(o + size_t(CAP) * 4);
        li = o;     o = align16(o + size_t(CAP) * 4);
        total = o;
    }
};

extern __shared__ __align__(16) unsigned char smem_raw[];

struct Smem {
    Slot* slot;          // [2] this CTA's exchange records (double-buffered)
    Slot* gath;          // [C] everyone's records after an exchange
    float* redf;         // [NW*4] per-warp scratch
    int* redi;           // [NW*4]
    int* misc;           // [32]
    uint32_t* segkey;    // [nsc] maximum order key per segment
    float* mass[3];      // [nsc] per-segment masses (current low / the two pivots)
    int* off;            // [nsc+1] per-segment counts / offsets / live-segment list
    float* lv;           // [CAP] compact list: values
    int* li;             // [CAP] compact list: token indices
    __device__ explicit Smem(const Layout& L) {
        slot = reinterpret_cast<Slot*>(smem_raw + L.slot);
        gath = reinterpret_cast<Slot*>(smem_raw + L.gath);
        redf = reinterpret_cast<float*>(smem_raw + L.redf);
        redi = reinterpret_cast<int*>(smem_raw + L.redi);
        misc = reinterpret_cast<int*>(smem_raw + L.misc);
        segkey = reinterpret_cast<uint32_t*>(smem_raw + L.segkey);
        mass[0] = reinterpret_cast<float*>(smem_raw + L.mass0);
        mass[1] = reinterpret_cast<float*>(smem_raw + L.mass1);
        mass[2] = reinterpret_cast<float*>(smem_raw + L.mass2);
        off = reinterpret_cast<int*>(smem_raw + L.off);
        lv = reinterpret_cast<float*>(smem_raw + L.lv);
        li = reinterpret_cast<int*>(smem_raw + L.li);
    }
};

// Which part of the row this CTA owns.
struct Geom {
    int V;
    int shift;     // log2(blocks per segment)
    int ns;        // segments per row
    int nsc_max;   // segments per CTA (the last CTA may own fewer)
    int s0;        // first segment of this CTA
    int nsc;       // segments owned by this CTA
    __device__ Geom(int V_, int shift_, int ns_, int nsc_max_, int rank)
        : V(V_), shift(shift_), ns(ns_), nsc_max(nsc_max_), s0(rank * nsc_max_) {
        nsc = max(0, min(nsc_max, ns - s0));
    }
    __device__ int seg_it() const { return 1 << shift; }
    // First element of block `it` of local segment `ls`, as seen by `lane`.
    __device__ int base(int ls, int it, int lane) const {
        return ((s0 + ls) << shift) * BLK + it * BLK + lane * 4;
    }
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
// CTA-wide barrier.
__device__ __forceinline__ void cluster_sync() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) { return __uint_as_float(ld_dsmem_u32(addr)); }

// ------------------------------------------------------------------ loads

// Elements [base, base+4) that straddle or pass the row end (or an unaligned row):
// element by element, `fill` past V.  Kept out of line: it is the cold path.
template <bool NC>
FS_NOINLINE __device__ float4 load4_tail(const float* __restrict__ row, int V, int base, float fill) {
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

// Visit this warp's segments in trips of T blocks (all loads of a trip in flight
// together).  Segments go to warps in runs of T / seg_it consecutive segments,
// round-robin.  live(ls) decides whether segment ls is read (warp-uniform);
// body(ls, it, base, x, on) sees block `it` of segment ls (x = fill when not live);
// done(ls, on) runs after the last block of segment ls.
template <int T, bool VEC, bool NC, typename LIVE, typename BODY, typename DONE>
__device__ __forceinline__ void visit(const float* __restrict__ row, const Geom& g, float fill, int warp, int lane,
                                      LIVE live, BODY body, DONE done) {
    static_assert(T >= (1 << MAX_SEG_SHIFT), "a trip must hold a whole segment");
    const int spt = T >> g.shift;
    const int mask = g.seg_it() - 1;
    const int per = spt << g.shift;  // blocks per trip actually used
    for (int first = warp * spt; first < g.nsc; first += NW * spt) {
        float4 v[T];
        bool on[T];
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const int ls = first + (j >> g.shift);
            on[j] = j < per && ls < g.nsc && live(ls);
            v[j] = on[j] ? load4<VEC, NC>(row, g.V, g.base(ls, j & mask, lane), fill)
                         : make_float4(fill, fill, fill, fill);
        }
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const int ls = first + (j >> g.shift);
            if (j < per && ls < g.nsc) {
                const int it = j & mask;
                body(ls, it, g.base(ls, it, lane), v[j], on[j]);
                if (it == mask) done(ls, on[j]);
            }
        }
    }
}

// ------------------------------------------------------------------ warp helpers

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

// Sum of a[0..n) in a fixed order: lane l accumulates a[l], a[l+32], ... in order,
// then the 32 lane sums are tree-reduced.  Warp-collective; identical in all lanes.
__device__ __forceinline__ float ordered_sum(const float* a, int n, int lane) {
    float acc = 0.f;
    for (int i = lane; i < n; i += 32) acc += a[i];
    return warp_sum(acc);
}
__device__ __forceinline__ uint32_t ordered_max_u(const uint32_t* a, int n, int lane) {
    uint32_t acc = 0;
    for (int i = lane; i < n; i += 32) acc = max(acc, a[i]);
    return warp_max_u(acc);
}

// ------------------------------------------------------------------ keys

// Order key of a probability: its bit pattern when positive, 0 for +-0.  For
// non-negative floats the integer order of the pattern is the numeric order
// ([drill] section 3).
__device__ __forceinline__ uint32_t prob_key(float x) { return x > 0.f ? __float_as_uint(x) : 0u; }

// Order-preserving key of a signed float ([drill] section 8: negative patterns sort
// backwards, so they are flipped; non-negative ones get the sign bit set).
__device__ __forceinline__ uint32_t logit_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

// ------------------------------------------------------------------ pass 1

// One streaming pass over this CTA's segments: per-segment maximum order key and
// (PROB) mass; per-lane positive count and a bad-value flag (NaN or negative for
// probabilities, NaN for logits).  Each warp keeps TRIP blocks in flight; the warp
// reductions of the TRIP blocks are interleaved.
template <bool VEC, bool NC, bool PROB>
__device__ __forceinline__ void pass1(const float* __restrict__ row, const Geom& g, uint32_t* segkey,
                                      float* segmass, int warp, int lane, int& pos, bool& bad) {
    const int spt = TRIP >> g.shift;
    const float fill = PROB ? 0.f : __int_as_float(0xff800000);
    for (int first = warp * spt; first < g.nsc; first += NW * spt) {
        float4 v[TRIP];
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            const int ls = first + (j >> g.shift);
            v[j] = ls < g.nsc ? load4<VEC, NC>(row, g.V, g.base(ls, j & (g.seg_it() - 1), lane), fill)
                              : make_float4(fill, fill, fill, fill);
        }
        float s[TRIP];
        uint32_t km[TRIP];
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            const int ls = first + (j >> g.shift);
            const int base = g.base(ls, j & (g.seg_it() - 1), lane);
            uint32_t k = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(v[j], q);
                if (PROB) {
                    bad |= !(x >= 0.f);
                    k = max(k, prob_key(x));
                    pos += x > 0.f;
                } else {
                    bad |= isnan(x);
                    k = max(k, (ls < g.nsc && base + q < g.V) ? logit_key(x) : 0u);
                }
            }
            km[j] = k;
            s[j] = PROB ? (v[j].x + v[j].y) + (v[j].z + v[j].w) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < TRIP; ++j) km[j] = __reduce_max_sync(FULL, km[j]);
        if (PROB) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TRIP; ++j) s[j] += __shfl_xor_sync(FULL, s[j], m);
        }
        // Lane t stores segment first + t (its blocks combined in block order).
        if (lane < spt && first + lane < g.nsc) {
            float ss = 0.f;
            uint32_t kk = 0;
#pragma unroll
            for (int j = 0; j < TRIP; ++j) {
                const bool mine = (j >> g.shift) == lane;
                ss += mine ? s[j] : 0.f;
                kk = mine ? max(kk, km[j]) : kk;
            }
            segkey[first + lane] = kk;
            if (PROB) segmass[first + lane] = ss;
        }
    }
}

// Fused (mass, count) above two pivots over the segments whose maximum exceeds p1
// (the rejection round's reduction, [blog] dual pivot).  Per-segment masses go to
// m1 / m2 (zero for skipped segments); per-lane counts accumulate into c1 / c2.
template <bool VEC, bool NC>
__device__ __forceinline__ void pivot_pass(const float* __restrict__ row, const Geom& g, const uint32_t* segkey,
                                           float p1, float p2, float* m1, float* m2, int warp, int lane, int& c1,
                                           int& c2) {
    const int spt = TRIP >> g.shift;
    const uint32_t kp1 = prob_key(p1);
    for (int first = warp * spt; first < g.nsc; first += NW * spt) {
        float4 v[TRIP];
        bool any = false;
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            const int ls = first + (j >> g.shift);
            const bool on = ls < g.nsc && segkey[ls] > kp1;
            any |= on;
            v[j] = on ? load4<VEC, NC>(row, g.V, g.base(ls, j & (g.seg_it() - 1), lane), 0.f)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float a[TRIP], b[TRIP];
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            float w1[4], w2[4];
            int cc = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(v[j], q);
                w1[q] = x > p1 ? x : 0.f;
                w2[q] = x > p2 ? x : 0.f;
                cc += int(x > p1) + (int(x > p2) << 16);
            }
            a[j] = (w1[0] + w1[1]) + (w1[2] + w1[3]);
            b[j] = (w2[0] + w2[1]) + (w2[2] + w2[3]);
            c1 += cc & 0xffff;
            c2 += cc >> 16;
        }
        if (any) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TRIP; ++j) {
                    a[j] += __shfl_xor_sync(FULL, a[j], m);
                    b[j] += __shfl_xor_sync(FULL, b[j], m);
                }
        }
        if (lane < spt && first + lane < g.nsc) {
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int j = 0; j < TRIP; ++j) {
                const bool mine = (j >> g.shift) == lane;
                sa += mine ? a[j] : 0.f;
                sb += mine ? b[j] : 0.f;
            }
            m1[first + lane] = sa;
            m2[first + lane] = sb;
        }
    }
}

// ------------------------------------------------------------------ cluster exchange

// Every CTA has filled the first `words` 32-bit words of slot[buf] (one thread).  After
// the barrier, the C slots are copied (one word per thread) into gath in rank order,
// and a CTA barrier publishes them.  Word i < 8 is f[i]; word 8 + i is u[i].
__device__ __forceinline__ void exchange(const Smem& sm, int buf, int C, int tid, int words = 20) {
    cluster_sync();
    for (int w = tid; w < C * words; w += NT) {
        const int c = w / words, o = w % words;
        const uint32_t a = map_rank(smem_u32(reinterpret_cast<const uint32_t*>(&sm.slot[buf]) + o), c);
        reinterpret_cast<uint32_t*>(&sm.gath[c])[o] = ld_dsmem_u32(a);
    }
    __syncthreads();
}

// ------------------------------------------------------------------ draws

// Inverse-transform locate inside one segment, warp-collective ([blog] inverse
// transform sampling; implementation details: a parallel float prefix sum need not be
// monotone, so the result is always forced onto an eligible token).  Eligible: x >
// low.  `t` is the target measured from the segment start.  Returns the first
// eligible element whose running sum exceeds t, else the segment's last eligible
// element.  The segment must hold an eligible element.
template <bool VEC, bool NC>
FS_NOINLINE __device__ void locate_in_segment(const float* __restrict__ row, const Geom& g, int ls, float low,
                                              float t, int lane, int* j_out, float* x_out) {
    float run = 0.f;
    int last_j = -1;
    float last_x = 0.f;
#pragma unroll 1
    for (int it = 0; it < g.seg_it(); ++it) {
        const int base = g.base(ls, it, lane);
        const float4 v = load4<VEC, NC>(row, g.V, base, 0.f);
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
            *j_out = __shfl_sync(FULL, base + pq, l);
            *x_out = __shfl_sync(FULL, q_at(v, pq), l);
            return;
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    *j_out = last_j;
    *x_out = last_x;
}

// First segment (local index) whose running mass over mass[0..n) exceeds t, with the
// mass before it in `before`; if none, the last segment with positive mass and
// `force_last` set.  Warp-collective.
FS_NOINLINE __device__ inline int locate_segment(const float* mass, int n, float t, int lane, float* before,
                                                 bool* force_last) {
    float run = 0.f;
    int last = -1;
    for (int base = 0; base < n; base += 32) {
        const float m = (base + lane < n) ? mass[base + lane] : 0.f;
        const float incl = warp_incl_scan(m, lane);
        const unsigned hit = __ballot_sync(FULL, m > 0.f && run + incl > t);
        const unsigned nz = __ballot_sync(FULL, m > 0.f);
        if (nz) last = base + 31 - __clz(nz);
        if (hit) {
            const int l = __ffs(hit) - 1;
            *before = run + __shfl_sync(FULL, incl - m, l);
            *force_last = false;
            return base + l;
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    *before = 0.f;
    *force_last = true;
    return last;
}

// Locate inside a compact list lv[0..n) (index order), eligible x > low.  Warp-collective.
FS_NOINLINE __device__ inline int locate_in_list(const float* lv, int n, float low, float t, int lane) {
    float run = 0.f;
    int last = -1;
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

// ------------------------------------------------------------------ compaction

// Ordered list of this CTA's segments whose maximum key is >= thr, into off[0..n).
// Block-collective; returns n.
FS_NOINLINE __device__ inline int live_segments(const Smem& sm, int nsc, uint32_t thr, int warp, int lane, int tid) {
    int out = 0;
    for (int base = 0; base < nsc; base += NT) {
        const int ls = base + tid;
        const bool live = ls < nsc && sm.segkey[ls] >= thr;
        const unsigned bal = __ballot_sync(FULL, live);
        if (lane == 0) sm.redi[warp] = __popc(bal);
        __syncthreads();
        int woff = out, chunk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int c = sm.redi[w];
            if (w < warp) woff += c;
            chunk += c;
        }
        __syncthreads();
        if (live) sm.off[woff + __popc(bal & ((1u << lane) - 1u))] = ls;
        out += chunk;
        __syncthreads();
    }
    return out;
}

// Collect, in index order, every element of this CTA's segments with key >= thr into
// lv/li (values, row indices), at most CAP of them.  Returns the exact count (which
// may exceed CAP; the caller treats that as overflow).  Block-collective.  Each
// batch of live segments is read once (one L2 round trip): counted, offsets scanned,
// then written from registers.
template <bool VEC, bool NC, typename KEYF>
FS_NOINLINE __device__ int compact_ge(const float* __restrict__ row, const Geom& g, uint32_t thr, KEYF keyf,
                                      float fill, const Smem& sm, int warp, int lane, int tid) {
    const int nlive = live_segments(sm, g.nsc, thr, warp, lane, tid);
    const int spt = TRIP >> g.shift;   // live segments a warp takes per batch
    int* cnt = sm.redi + 2 * NW;       // per-warp counts of the current batch (NW entries)
    int total = 0;
    for (int b0 = 0; b0 < nlive; b0 += NW * spt) {
        float4 v[TRIP];
        int c = 0;
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            const int li = b0 + warp * spt + (j >> g.shift);
            const bool on = li < nlive;
            const int ls = on ? sm.off[li] : 0;
            v[j] = on ? load4<VEC, NC>(row, g.V, g.base(ls, j & (g.seg_it() - 1), lane), fill)
                      : make_float4(fill, fill, fill, fill);
            if (on) {
                const int base = g.base(ls, j & (g.seg_it() - 1), lane);
#pragma unroll
                for (int q = 0; q < 4; ++q) c += __popc(__ballot_sync(FULL, keyf(q_at(v[j], q)) >= thr && base + q < g.V));
            }
        }
        if (lane == 0) cnt[warp] = c;
        __syncthreads();
        int pos = total, chunk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (w < warp) pos += cnt[w];
            chunk += cnt[w];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < TRIP; ++j) {
            const int li = b0 + warp * spt + (j >> g.shift);
            if (li < nlive) {
                const int ls = sm.off[li];
                const int base = g.base(ls, j & (g.seg_it() - 1), lane);
                bool keep[4];
                int k = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    keep[q] = keyf(q_at(v[j], q)) >= thr && base + q < g.V;
                    k += keep[q];
                }
                const int incl = warp_incl_scan_i(k, lane);
                int p = pos + incl - k;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (keep[q]) {
                        if (p < CAP) {
                            sm.lv[p] = q_at(v[j], q);
                            sm.li[p] = base + q;
                        }
                        ++p;
                    }
                }
                pos += __shfl_sync(FULL, incl, 31);
            }
        }
        total += chunk;
    }
    __syncthreads();
    return total;
}

// Rank 0: append the lists of ranks 1..C-1 (lengths in gath[c].u[cnt_idx]) after its
// own, keeping only entries with key >= keep_thr, in rank then index order.  Returns
// the new length (at most CAP).  Block-collective on rank 0.  Entries are compacted
// in place: a write never lands past the entry being read.
template <typename KEYF>
FS_NOINLINE __device__ int gather_lists(const Smem& sm, int C, int cnt_idx, uint32_t keep_thr, KEYF keyf, int warp,
                                        int lane, int tid) {
    int total = 0;
    for (int c = 0; c < C; ++c) total += int(sm.gath[c].u[cnt_idx]);
    int out = 0;
    for (int base = 0; base < total; base += NT) {
        const int e = base + tid;
        float v = 0.f;
        int ix = 0;
        bool keep = false;
        if (e < total) {
            int c = 0, acc = 0;
            while (c < C - 1 && e >= acc + int(sm.gath[c].u[cnt_idx])) {
                acc += int(sm.gath[c].u[cnt_idx]);
                ++c;
            }
            const int le = e - acc;
            if (c == 0) {
                v = sm.lv[le];
                ix = sm.li[le];
            } else {
                v = ld_dsmem_f32(map_rank(smem_u32(sm.lv + le), c));
                ix = int(ld_dsmem_u32(map_rank(smem_u32(sm.li + le), c)));
            }
            keep = keyf(v) >= keep_thr;
        }
        const unsigned bal = __ballot_sync(FULL, keep);
        if (lane == 0) sm.redi[warp] = __popc(bal);
        __syncthreads();
        int woff = out;
        int chunk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int n = sm.redi[w];
            if (w < warp) woff += n;
            chunk += n;
        }
        const int p = woff + __popc(bal & ((1u << lane) - 1u));
        if (keep && p < CAP) {
            sm.lv[p] = v;
            sm.li[p] = ix;
        }
        out += chunk;
        __syncthreads();
    }
    return min(out, CAP);
}

// Largest key t among the keys of lv[0..n) with #{key >= t} >= k; 0 if none.
// Block-collective (rank counting; the list is short).
template <typename KEYF>
FS_NOINLINE __device__ uint32_t kth_key_in_list(const Smem& sm, int n, int k, KEYF keyf, int warp, int lane, int tid) {
    uint32_t best = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t ki = keyf(sm.lv[i]);
        int ge = 0;
        for (int j = 0; j < n; ++j) ge += (keyf(sm.lv[j]) >= ki);
        if (ge >= k) best = max(best, ki);
    }
    best = warp_max_u(best);
    if (lane == 0) sm.redi[warp] = int(best);
    __syncthreads();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = max(r, uint32_t(sm.redi[w]));
    __syncthreads();
    return r;
}

// Largest value t among a[0..n) with #{a >= t} >= k; 0 if none.  Block-collective.
FS_NOINLINE __device__ inline uint32_t kth_in_array(const uint32_t* a, int n, int k, const Smem& sm, int warp,
                                                    int lane, int tid) {
    uint32_t best = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t ki = a[i];
        int ge = 0;
        for (int j = 0; j < n; ++j) ge += (a[j] >= ki);
        if (ge >= k) best = max(best, ki);
    }
    best = warp_max_u(best);
    if (lane == 0) sm.redi[warp] = int(best);
    __syncthreads();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = max(r, uint32_t(sm.redi[w]));
    __syncthreads();
    return r;
}

// In-place, order-preserving filter of lv/li[0..n) to key >= t by one warp.
// Returns the new length (warp-uniform).
template <typename KEYF>
FS_NOINLINE __device__ int filter_list_warp(const Smem& sm, int n, uint32_t t, KEYF keyf, int lane) {
    int w = 0;
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const bool keep = i < n && keyf(sm.lv[i]) >= t;
        const float xv = keep ? sm.lv[i] : 0.f;
        const int xi = keep ? sm.li[i] : 0;
        const unsigned bal = __ballot_sync(FULL, keep);
        const int pos = w + __popc(bal & ((1u << lane) - 1u));
        __syncwarp();
        if (keep) {
            sm.lv[pos] = xv;
            sm.li[pos] = xi;
        }
        __syncwarp();
        w += __popc(bal);
    }
    return w;
}

// ------------------------------------------------------------------ bisection

// Interval of a threshold search over order keys ([drill] sections 2-3: bisection on a
// monotone count or mass, done on the integer bit pattern so that it ends exactly on
// an existing value).  Invariant: crit(lo) holds and crit(hi) does not, where
// crit(t) = count(key >= t) >= k  or  mass(key >= t) >= target.  Done when
// hi = lo + 1; then lo is the threshold.
struct Bisect {
    uint64_t lo, hi;
    int cnt_lo;       // count(key >= lo)
    float mass_lo;    // mass(key >= lo) (probabilities only)
};

// Drive the search to the end with passes of three pivots ([drill] section 5: the
// production kernel tries several pivots per pass and stops once a single value is
// left).  Each pass counts (and sums, MASS) the elements at or above each pivot and
// records the smallest and largest key inside each of the four sub-intervals, so the
// next interval shrinks to the keys that exist in it.  All CTAs of the cluster call
// it with identical state and leave with identical results.  At most 40 passes.
template <bool VEC, bool NC, bool MASS, typename KEYF>
FS_NOINLINE __device__ void bisect_run(const float* __restrict__ row, const Geom& g, Bisect* stp, int kcrit,
                                       float target, KEYF keyf, float fill, const Smem& sm, int* bufp, int C,
                                       int warp, int lane, int tid) {
    Bisect st = *stp;
    int buf = *bufp;
    for (int iter = 0; iter < 40 && st.hi - st.lo > 1; ++iter) {
        const uint64_t d = st.hi - st.lo;
        uint32_t piv[3];
        if (d >= 4) {
#pragma unroll
            for (int i = 0; i < 3; ++i) piv[i] = uint32_t(st.lo + (d * uint64_t(i + 1)) / 4);
        } else {
            piv[0] = uint32_t(st.lo + 1);
            piv[1] = uint32_t(d == 3 ? st.lo + 2 : st.hi);
            piv[2] = uint32_t(st.hi);
        }
        const uint64_t lo = st.lo, hi = st.hi;
        float m[3] = {0.f, 0.f, 0.f};
        int c[3] = {0, 0, 0};
        uint32_t mn[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        uint32_t mx[4] = {0u, 0u, 0u, 0u};
        visit<4, VEC, NC>(
            row, g, fill, warp, lane, [&](int ls) { return uint64_t(sm.segkey[ls]) >= lo; },
            [&](int, int, int base, float4 x, bool on) {
                if (!on) return;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float xv = q_at(x, q);
                    const uint32_t key = keyf(xv);
                    const bool inr = base + q < g.V;
                    const bool g0 = inr && key >= piv[0], g1 = inr && key >= piv[1], g2 = inr && key >= piv[2];
                    if (MASS) {
                        m[0] += g0 ? xv : 0.f;
                        m[1] += g1 ? xv : 0.f;
                        m[2] += g2 ? xv : 0.f;
                    }
                    c[0] += g0;
                    c[1] += g1;
                    c[2] += g2;
                    const bool inlo = inr && uint64_t(key) >= lo && uint64_t(key) < hi;
                    const int bkt = int(g0) + int(g1) + int(g2);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const bool sel = inlo && t == bkt;
                        mn[t] = sel ? min(mn[t], key) : mn[t];
                        mx[t] = sel ? max(mx[t], key) : mx[t];
                    }
                }
            },
            [&](int, bool) {});
        // Warp, then block, then cluster reductions (fixed order).
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            m[i] = warp_sum(m[i]);
            c[i] = warp_sum_i(c[i]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            mn[t] = warp_min_u(mn[t]);
            mx[t] = warp_max_u(mx[t]);
        }
        if (lane == 0) {
            for (int i = 0; i < 3; ++i) {
                sm.redf[warp * 4 + i] = m[i];
                sm.redi[warp * 4 + i] = c[i];
            }
        }
        __syncthreads();
        if (tid == 0) {
            for (int i = 0; i < 3; ++i) {
                float a = 0.f;
                uint32_t b = 0;
                for (int w = 0; w < NW; ++w) {
                    a += sm.redf[w * 4 + i];
                    b += uint32_t(sm.redi[w * 4 + i]);
                }
                sm.slot[buf].f[i] = a;
                sm.slot[buf].u[i] = b;
            }
        }
        __syncthreads();
        if (lane == 0) {
            for (int t = 0; t < 4; ++t) {
                sm.redi[warp * 4 + t] = int(mn[t]);
                reinterpret_cast<uint32_t*>(sm.redf)[warp * 4 + t] = mx[t];
            }
        }
        __syncthreads();
        if (tid == 0) {
            for (int t = 0; t < 4; ++t) {
                uint32_t a = 0xffffffffu, b = 0u;
                for (int w = 0; w < NW; ++w) {
                    a = min(a, uint32_t(sm.redi[w * 4 + t]));
                    b = max(b, reinterpret_cast<const uint32_t*>(sm.redf)[w * 4 + t]);
                }
                sm.slot[buf].u[3 + t] = a;
                sm.slot[buf].u[7 + t] = b;
            }
        }
        exchange(sm, buf, C, tid);
        buf ^= 1;
        float mass[3] = {0.f, 0.f, 0.f};
        int cnt[3] = {0, 0, 0};
        uint32_t kmin[4], kmax[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            kmin[t] = 0xffffffffu;
            kmax[t] = 0u;
        }
        for (int cc = 0; cc < C; ++cc) {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                mass[i] += sm.gath[cc].f[i];
                cnt[i] += int(sm.gath[cc].u[i]);
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                kmin[t] = min(kmin[t], sm.gath[cc].u[3 + t]);
                kmax[t] = max(kmax[t], sm.gath[cc].u[7 + t]);
            }
        }
        // crit is monotone in the pivot: take the largest pivot where it holds.
        int best = -1;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            if (uint64_t(piv[i]) < hi) {
                const bool ok = MASS ? (mass[i] >= target) : (cnt[i] >= kcrit);
                if (ok) best = i;
            }
        }
        uint64_t nlo = lo, nhi = hi;
        int bkt = 0;
        if (best >= 0) {
            nlo = piv[best];
            st.cnt_lo = cnt[best];
            st.mass_lo = mass[best];
            bkt = best + 1;
        }
        if (best + 1 < 3 && uint64_t(piv[best + 1]) < hi) nhi = piv[best + 1];
        if (kmin[bkt] <= kmax[bkt]) {  // keys present in the new interval
            nlo = max(nlo, uint64_t(kmin[bkt]));
            nhi = min(nhi, uint64_t(kmax[bkt]) + 1);
        }
        st.lo = nlo;
        st.hi = nhi;
        __syncthreads();  // gath is rewritten by the next exchange
    }
    *stp = st;
    *bufp = buf;
}

// Count and mass (probabilities, x > 0) of key >= t over this CTA's segments, then
// cluster-wide.  When seg_mass is given the per-segment masses are stored there and
// the CTA mass is their ordered sum (what a later draw scans); per_rank (shared
// memory, nullable) receives the C per-CTA masses.
template <bool VEC, bool NC, typename KEYF>
FS_NOINLINE __device__ void mass_count_ge(const float* __restrict__ row, const Geom& g, uint32_t t, KEYF keyf,
                                          float* seg_mass, const Smem& sm, int* bufp, int C, int warp, int lane,
                                          int tid, float* mass_out, int* cnt_out, float* per_rank) {
    float wm = 0.f, ms = 0.f;
    int wc = 0;
    visit<4, VEC, NC>(
        row, g, 0.f, warp, lane, [&](int ls) { return sm.segkey[ls] >= t; },
        [&](int, int it, int base, float4 x, bool on) {
            if (it == 0) ms = 0.f;
            if (!on) return;
            float s = 0.f;
            int c = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xv = q_at(x, q);
                const bool gq = keyf(xv) >= t && xv > 0.f && base + q < g.V;
                s += gq ? xv : 0.f;
                c += gq;
            }
            ms += warp_sum(s);
            wc += warp_sum_i(c);
        },
        [&](int ls, bool) {
            if (seg_mass && lane == 0) seg_mass[ls] = ms;
            wm += ms;
        });
    if (lane == 0) {
        sm.redf[warp] = wm;
        sm.redi[warp] = wc;
    }
    __syncthreads();
    const int buf = *bufp;
    if (warp == 0) {
        float s = 0.f;
        if (seg_mass) {
            s = ordered_sum(seg_mass, g.nsc, lane);
        } else {
#pragma unroll
            for (int w = 0; w < NW; ++w) s += sm.redf[w];
        }
        int n = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) n += sm.redi[w];
        if (lane == 0) {
            sm.slot[buf].f[0] = s;
            sm.slot[buf].u[0] = uint32_t(n);
        }
    }
    exchange(sm, buf, C, tid);
    *bufp = buf ^ 1;
    float mass = 0.f;
    int cnt = 0;
    for (int c = 0; c < C; ++c) {
        mass += sm.gath[c].f[0];
        cnt += int(sm.gath[c].u[0]);
    }
    if (per_rank && tid < C) per_rank[tid] = sm.gath[tid].f[0];
    __syncthreads();
    *mass_out = mass;
    *cnt_out = cnt;
}

}  // namespace fsd
