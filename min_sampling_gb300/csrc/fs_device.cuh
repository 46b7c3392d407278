// Device building blocks shared by the sampling and filter kernels (sm_103a).
//
// Execution model: one thread-block cluster of C CTAs per row, rank 0 the leader.
// A row is cut into segments of 128 * 2^shift elements (128 = one float4 per lane of
// a warp).  Every CTA streams a contiguous share of the segments from HBM exactly
// once (pass 1), and writes each segment's maximum order key and mass straight into
// the leader's shared memory (distributed shared memory stores), so that after one
// cluster barrier the leader holds the whole row's segment table.  From there the
// leader drives the rest: it finishes alone when little data is left to touch (the
// top-k candidates, a compact list of surviving tokens), and otherwise sends the
// other CTAs commands (a two-pivot reduction pass, a three-pivot bisection pass, a
// masked write) through their shared memory, each command bracketed by two cluster
// barriers.  Every CTA executes the same sequence of cluster barriers: the peers
// follow the leader's commands until an EXIT command.
//
// Code size is kept small on purpose: the work after pass 1 runs once per CTA, from
// a cold instruction cache, on every SM at the same moment.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define FS_NOINLINE __noinline__

namespace fsd {

constexpr int NT = 256;                 // threads per CTA
constexpr int NW = NT / 32;             // warps per CTA
constexpr int BLK = 128;                // elements per block (one float4 per lane)
constexpr int TB = 4;                   // blocks per trip (double-buffered in pass 1)
constexpr int MAX_SEG_SHIFT = 2;        // at most 4 blocks per segment (V <= 2^21)
constexpr int NS_TARGET = 4096;         // segments per row (longer rows use longer segments)
constexpr int CAP = 2048;               // compact-list capacity (leader)
constexpr int R_MAX = 256;              // rejection rounds before a row is invalid
constexpr int MAX_CLUSTER = 8;
constexpr unsigned FULL = 0xffffffffu;

// Commands from the leader to the other CTAs of the cluster.
enum : int { CMD_EXIT = 0, CMD_PIVOT2 = 1, CMD_BISECT = 2, CMD_MASSGE = 3, CMD_WRITE = 4 };

// ------------------------------------------------------------------ geometry

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Smallest shift s with ceil(V / (BLK << s)) <= NS_TARGET.
__host__ __device__ inline int seg_shift_for(int V) {
    int s = 0;
    while (s < MAX_SEG_SHIFT && (V + (BLK << s) - 1) / (BLK << s) > NS_TARGET) ++s;
    return s;
}

// A command (written by the leader into every CTA's copy).
struct Ctl {
    int cmd;
    int ia, ib;            // PIVOT2: which mass arrays receive the per-segment masses
    int flag;              // WRITE: row valid
    float f[4];            // pivots / denominator
    uint32_t u[4];         // key pivots / threshold; u[3] = interval low (BISECT)
    uint32_t hi_lo, hi_hi; // BISECT: 64-bit interval high
};

// One CTA's partial results, in the leader's shared memory (one record per rank).
struct Part {
    float f[4];
    uint32_t u[12];
};

// Byte offsets of the dynamic shared-memory carve-up for `ns` segments per row.
struct Layout {
    size_t ctl, part, red, segkey, mass0, mass1, mass2, list, lv, li, total;
    __host__ __device__ explicit Layout(int ns) {
        size_t o = 0;
        ctl = o;    o = align16(o + sizeof(Ctl));
        part = o;   o = align16(o + MAX_CLUSTER * sizeof(Part));
        red = o;    o = align16(o + 64 * sizeof(int));
        segkey = o; o = align16(o + size_t(ns) * 4);
        mass0 = o;  o = align16(o + size_t(ns) * 4);
        mass1 = o;  o = align16(o + size_t(ns) * 4);
        mass2 = o;  o = align16(o + size_t(ns) * 4);
        list = o;   o = align16(o + size_t(ns + 1) * 4);
        lv = o;     o = align16(o + size_t(CAP) * 4);
        li = o;     o = align16(o + size_t(CAP) * 4);
        total = o;
    }
};

extern __shared__ __align__(16) unsigned char smem_raw[];

struct Smem {
    Ctl* ctl;            // the current command
    Part* part;          // [MAX_CLUSTER] partial results (leader)
    int* red;            // [64] block-reduction scratch
    uint32_t* segkey;    // [ns] maximum order key per segment (row-wide on the leader)
    float* mass[3];      // [ns] per-segment masses (row-wide on the leader)
    int* list;           // [ns+1] live-segment list / offsets (leader)
    float* lv;           // [CAP] compact list: values (leader)
    int* li;             // [CAP] compact list: token indices (leader)
    __device__ explicit Smem(int ns) {
        const Layout L(ns);
        ctl = reinterpret_cast<Ctl*>(smem_raw + L.ctl);
        part = reinterpret_cast<Part*>(smem_raw + L.part);
        red = reinterpret_cast<int*>(smem_raw + L.red);
        segkey = reinterpret_cast<uint32_t*>(smem_raw + L.segkey);
        mass[0] = reinterpret_cast<float*>(smem_raw + L.mass0);
        mass[1] = reinterpret_cast<float*>(smem_raw + L.mass1);
        mass[2] = reinterpret_cast<float*>(smem_raw + L.mass2);
        list = reinterpret_cast<int*>(smem_raw + L.list);
        lv = reinterpret_cast<float*>(smem_raw + L.lv);
        li = reinterpret_cast<int*>(smem_raw + L.li);
    }
};

// The row, its segmentation and this CTA's share.  Segment indices are row-wide.
struct Geom {
    int V;
    int shift;     // log2(blocks per segment)
    int ns;        // segments per row
    int s0, s1;    // this CTA's segments [s0, s1)
    __device__ Geom(int V_, int shift_, int ns_, int nsc, int rank) : V(V_), shift(shift_), ns(ns_) {
        s0 = min(ns, rank * nsc);
        s1 = min(ns, s0 + nsc);
    }
    __device__ int seg_it() const { return 1 << shift; }
    // First element of block `it` of segment `s`, as seen by `lane`.
    __device__ int base(int s, int it, int lane) const { return ((s << shift) + it) * BLK + lane * 4; }
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
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Store a word into the leader's copy of a shared-memory location (local store on the
// leader itself).
__device__ __forceinline__ void put_leader(void* local_addr, uint32_t v, bool leader) {
    if (leader) {
        *reinterpret_cast<uint32_t*>(local_addr) = v;
    } else {
        st_dsmem_u32(map_rank(smem_u32(local_addr), 0), v);
    }
}

// ------------------------------------------------------------------ loads

// Elements [base, base+4) that straddle the row end, or of an unaligned row: element
// by element, `fill` past V.  Out of line: the cold path.
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

// ------------------------------------------------------------------ warp / block helpers

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

// Sum of a[0..n) in a fixed order, by the whole CTA: warp w sums its contiguous range
// (lane-strided, then a tree), the NW range sums are added in warp order.  Every
// thread gets the same value.  Uses red[0..NW) and two CTA barriers.
FS_NOINLINE __device__ inline float block_ordered_sum(const float* a, int n, int* red, int warp, int lane) {
    int r0, r1;
    warp_range(n, warp, r0, r1);
    float acc = 0.f;
    for (int i = r0 + lane; i < r1; i += 32) acc += a[i];
    acc = warp_sum(acc);
    float* rf = reinterpret_cast<float*>(red);
    if (lane == 0) rf[warp] = acc;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += rf[w];
    __syncthreads();
    return s;
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

// One streaming pass over this CTA's segments.  Warp w takes a contiguous range of
// them and reads it in trips of TB blocks with the next trip's loads in flight while
// the current trip is reduced.  For every segment: the maximum order key and (PROB)
// the mass, stored locally (segment key) and into the leader's table.  Per lane: the
// positive count and a bad-value flag (NaN or negative for probabilities, NaN for
// logits).
template <bool VEC, bool NC, bool PROB>
__device__ __forceinline__ void pass1(const float* __restrict__ row, const Geom& g, const Smem& sm, bool leader,
                                      int warp, int lane, int& pos, bool& bad) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const int nblk = (r1 - r0) << g.shift;
    const int mask = g.seg_it() - 1;
    const float fill = PROB ? 0.f : __int_as_float(0xff800000);
    float4 A[TB], Bv[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j)
        A[j] = j < nblk ? load4<VEC, NC>(row, g.V, g.base(r0 + (j >> g.shift), j & mask, lane), fill)
                        : make_float4(fill, fill, fill, fill);
    for (int b0 = 0; b0 < nblk; b0 += TB) {
        const int nb = b0 + TB;
#pragma unroll
        for (int j = 0; j < TB; ++j)
            Bv[j] = nb + j < nblk
                        ? load4<VEC, NC>(row, g.V, g.base(r0 + ((nb + j) >> g.shift), (nb + j) & mask, lane), fill)
                        : make_float4(fill, fill, fill, fill);
        float s[TB];
        uint32_t km[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int blk = b0 + j;
            const int base = g.base(r0 + (blk >> g.shift), blk & mask, lane);
            uint32_t k = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(A[j], q);
                if (PROB) {
                    bad |= !(x >= 0.f);
                    k = max(k, prob_key(x));
                    pos += x > 0.f;
                } else {
                    bad |= isnan(x);
                    k = max(k, (blk < nblk && base + q < g.V) ? logit_key(x) : 0u);
                }
            }
            km[j] = __reduce_max_sync(FULL, k);
            s[j] = PROB ? (A[j].x + A[j].y) + (A[j].z + A[j].w) : 0.f;
        }
        if (PROB) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TB; ++j) s[j] += __shfl_xor_sync(FULL, s[j], m);
        }
        // Lane t stores segment (b0 >> shift) + t, its blocks combined in order.
        const int nseg = TB >> g.shift;
        const int sg = r0 + (b0 >> g.shift) + lane;
        if (lane < nseg && sg < r1) {
            float ss = 0.f;
            uint32_t kk = 0;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const bool mine = (j >> g.shift) == lane;
                ss += mine ? s[j] : 0.f;
                kk = mine ? max(kk, km[j]) : kk;
            }
            sm.segkey[sg] = kk;
            if (!leader) put_leader(&sm.segkey[sg], kk, false);
            if (PROB) put_leader(&sm.mass[0][sg], __float_as_uint(ss), leader);
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) A[j] = Bv[j];
    }
}

// The rejection round's fused reduction ([blog] dual pivot) over this CTA's segments
// whose maximum exceeds p1: per segment the mass above p1 and above p2 (stored into
// the leader's mass[ia] / mass[ib]; zero for skipped segments); per lane the counts.
template <bool VEC, bool NC>
FS_NOINLINE __device__ void pivot_pass(const float* __restrict__ row, const Geom& g, const Smem& sm, bool leader,
                                       float p1, float p2, int ia, int ib, int warp, int lane, int* c1o, int* c2o) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const uint32_t kp1 = prob_key(p1);
    const int mask = g.seg_it() - 1;
    int c1 = 0, c2 = 0;
    for (int b0 = 0; b0 < ((r1 - r0) << g.shift); b0 += TB) {
        float4 v[TB];
        bool any = false;
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int blk = b0 + j;
            const int sg = r0 + (blk >> g.shift);
            const bool on = sg < r1 && sm.segkey[sg] > kp1;
            any |= on;
            v[j] = on ? load4<VEC, NC>(row, g.V, g.base(sg, blk & mask, lane), 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float a[TB], b[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            float w1[4], w2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(v[j], q);
                w1[q] = x > p1 ? x : 0.f;
                w2[q] = x > p2 ? x : 0.f;
                c1 += x > p1;
                c2 += x > p2;
            }
            a[j] = (w1[0] + w1[1]) + (w1[2] + w1[3]);
            b[j] = (w2[0] + w2[1]) + (w2[2] + w2[3]);
        }
        if (any) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TB; ++j) {
                    a[j] += __shfl_xor_sync(FULL, a[j], m);
                    b[j] += __shfl_xor_sync(FULL, b[j], m);
                }
        }
        const int nseg = TB >> g.shift;
        const int sg = r0 + (b0 >> g.shift) + lane;
        if (lane < nseg && sg < r1) {
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const bool mine = (j >> g.shift) == lane;
                sa += mine ? a[j] : 0.f;
                sb += mine ? b[j] : 0.f;
            }
            put_leader(&sm.mass[ia][sg], __float_as_uint(sa), leader);
            put_leader(&sm.mass[ib][sg], __float_as_uint(sb), leader);
        }
    }
    *c1o = warp_sum_i(c1);
    *c2o = warp_sum_i(c2);
}

// ------------------------------------------------------------------ leader-side helpers

// Ordered list of the segments s in [0, ns) with segkey[s] >= thr, into list[0..n).
// Block-collective; returns n.
FS_NOINLINE __device__ inline int live_list(const Smem& sm, int ns, uint32_t thr, int warp, int lane) {
    int r0, r1;
    warp_range(ns, warp, r0, r1);
    int cnt = 0;
    for (int base = r0; base < r1; base += 32) {
        const int i = base + lane;
        cnt += __popc(__ballot_sync(FULL, i < r1 && sm.segkey[i] >= thr));
    }
    if (lane == 0) sm.red[warp] = cnt;
    __syncthreads();
    int off = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) off += sm.red[w];
        total += sm.red[w];
    }
    for (int base = r0; base < r1; base += 32) {
        const int i = base + lane;
        const bool live = i < r1 && sm.segkey[i] >= thr;
        const unsigned bal = __ballot_sync(FULL, live);
        if (live) sm.list[off + __popc(bal & ((1u << lane) - 1u))] = i;
        off += __popc(bal);
    }
    __syncthreads();
    return total;
}

// Leader: read the listed segments (list[0..nlive), in order) and collect, in index
// order, every element with key >= thr into lv/li.  Returns the exact count (the
// list holds at most CAP; more means overflow).  Each warp takes TB blocks of listed
// segments per batch, so a batch is one L2 round trip.  Block-collective.
template <bool VEC, bool NC, typename KEYF>
FS_NOINLINE __device__ int collect(const float* __restrict__ row, const Geom& g, const Smem& sm, int nlive,
                                   uint32_t thr, KEYF keyf, float fill, int warp, int lane) {
    constexpr int CB = 8;              // blocks per warp per batch
    const int spw = CB >> g.shift;   // listed segments per warp per batch
    const int mask = g.seg_it() - 1;
    int total = 0;
    for (int b0 = 0; b0 < nlive; b0 += NW * spw) {
        float4 v[CB];
        int c = 0;
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int li = b0 + warp * spw + (j >> g.shift);
            const bool on = li < nlive;
            const int sg = on ? sm.list[li] : 0;
            v[j] = on ? load4<VEC, NC>(row, g.V, g.base(sg, j & mask, lane), fill)
                      : make_float4(fill, fill, fill, fill);
        }
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int li = b0 + warp * spw + (j >> g.shift);
            if (li < nlive) {
                const int base = g.base(sm.list[li], j & mask, lane);
#pragma unroll
                for (int q = 0; q < 4; ++q) c += __popc(__ballot_sync(FULL, keyf(q_at(v[j], q)) >= thr && base + q < g.V));
            }
        }
        if (lane == 0) sm.red[warp] = c;
        __syncthreads();
        int pos = total, chunk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (w < warp) pos += sm.red[w];
            chunk += sm.red[w];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int li = b0 + warp * spw + (j >> g.shift);
            if (li < nlive) {
                const int base = g.base(sm.list[li], j & mask, lane);
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

// Largest key t among the keys of lv[0..n) with #{key >= t} >= k; 0 if none.
// Block-collective (rank counting; the list is short).
template <typename KEYF>
FS_NOINLINE __device__ uint32_t kth_key_in_list(const Smem& sm, int n, int k, KEYF keyf, int warp, int lane,
                                                int tid) {
    uint32_t best = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t ki = keyf(sm.lv[i]);
        int ge = 0;
        for (int j = 0; j < n; ++j) ge += (keyf(sm.lv[j]) >= ki);
        if (ge >= k) best = max(best, ki);
    }
    best = warp_max_u(best);
    if (lane == 0) sm.red[warp] = int(best);
    __syncthreads();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = max(r, uint32_t(sm.red[w]));
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

// ------------------------------------------------------------------ draws

// Inverse-transform locate inside one segment, warp-collective ([blog] inverse
// transform sampling; implementation details: a parallel float prefix sum need not be
// monotone, so the result is always forced onto an eligible token).  Eligible: x >
// low.  `t` is the target measured from the segment start.  Returns the first
// eligible element whose running sum exceeds t, else the segment's last eligible
// element.  The segment must hold an eligible element.
template <bool VEC, bool NC>
FS_NOINLINE __device__ void locate_in_segment(const float* __restrict__ row, const Geom& g, int s, float low, float t,
                                              int lane, int* j_out, float* x_out) {
    float run = 0.f;
    int last_j = -1;
    float last_x = 0.f;
    for (int it = 0; it < g.seg_it(); ++it) {
        const int base = g.base(s, it, lane);
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

// The segment holding target t in the running mass over mass[0..n), by the whole CTA:
// warp range sums (the same grouping block_ordered_sum uses), the range holding t,
// then the segment inside it.  If no running mass exceeds t (rounding), the last
// segment with positive mass.  Returns the segment and the mass before it; every
// thread gets them.  Block-collective.
FS_NOINLINE __device__ inline int locate_segment_block(const float* mass, int n, float t, int* red, int warp,
                                                       int lane, float* before_out) {
    int r0, r1;
    warp_range(n, warp, r0, r1);
    float acc = 0.f;
    for (int i = r0 + lane; i < r1; i += 32) acc += mass[i];
    acc = warp_sum(acc);
    float* rf = reinterpret_cast<float*>(red);
    if (lane == 0) rf[warp] = acc;
    __syncthreads();
    int res = -1;
    float before = 0.f;
    if (warp == 0) {
        // Range holding t (guarded: the last range with positive mass).
        float run = 0.f, lastb = 0.f;
        int w_hit = -1, w_last = -1;
        for (int w = 0; w < NW; ++w) {
            const float m = rf[w];
            if (m > 0.f) {
                if (w_hit < 0 && run + m > t) {
                    w_hit = w;
                    before = run;
                }
                w_last = w;
                lastb = run;
            }
            run += m;
        }
        bool force = false;
        if (w_hit < 0) {
            w_hit = w_last;
            before = lastb;
            force = true;
        }
        if (w_hit >= 0) {
            int a0, a1;
            warp_range(n, w_hit, a0, a1);
            float tt = force ? __int_as_float(0x7f800000) : t - before;
            float r = 0.f;
            int last = -1;
            float last_before = 0.f;
            for (int base = a0; base < a1; base += 32) {
                const float m = (base + lane < a1) ? mass[base + lane] : 0.f;
                const float incl = warp_incl_scan(m, lane);
                const unsigned hit = __ballot_sync(FULL, m > 0.f && r + incl > tt);
                const unsigned nz = __ballot_sync(FULL, m > 0.f);
                if (nz) {
                    const int l = 31 - __clz(nz);
                    last = base + l;
                    last_before = r + __shfl_sync(FULL, incl - m, l);
                }
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    res = base + l;
                    before += r + __shfl_sync(FULL, incl - m, l);
                    break;
                }
                r += __shfl_sync(FULL, incl, 31);
            }
            if (res < 0) {
                res = last;
                before += last_before;
            }
        }
        if (lane == 0) {
            red[NW] = res;
            rf[NW + 1] = before;
        }
    }
    __syncthreads();
    res = red[NW];
    before = rf[NW + 1];
    __syncthreads();
    *before_out = before;
    return res;
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

// ------------------------------------------------------------------ commands

// Leader: publish a command into every CTA's Ctl (DSMEM stores), then the cluster
// barrier after which the peers read it.  Block-collective on the leader.
__device__ __forceinline__ void send_command(const Smem& sm, const Ctl& c, int C, int tid) {
    constexpr int W = sizeof(Ctl) / 4;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&c);
    if (tid < C * W) {
        const int r = tid / W, o = tid % W;
        uint32_t* dst = reinterpret_cast<uint32_t*>(sm.ctl) + o;
        if (r == 0) {
            *dst = src[o];
        } else {
            st_dsmem_u32(map_rank(smem_u32(dst), r), src[o]);
        }
    }
    cluster_sync();
}

// A three-pivot bisection pass ([drill] sections 3-5) over this CTA's segments whose
// maximum key is >= lo: count and (MASS) mass of keys >= each pivot, and per
// sub-interval [lo,p0) [p0,p1) [p1,p2) [p2,hi) the smallest and largest key present.
// The CTA's record goes to the leader's part[rank]: f[0..2] masses, u[0..2] counts,
// u[3..6] min keys, u[7..10] max keys.  Block-collective.
template <bool VEC, bool NC, bool MASS, typename KEYF>
FS_NOINLINE __device__ void bisect_pass(const float* __restrict__ row, const Geom& g, const Smem& sm, bool leader,
                                        int rank, uint64_t lo, uint64_t hi, const uint32_t* piv, KEYF keyf,
                                        float fill, int warp, int lane, int tid) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const int mask = g.seg_it() - 1;
    const uint32_t p0 = piv[0], p1 = piv[1], p2 = piv[2];
    float m[3] = {0.f, 0.f, 0.f};
    int c[3] = {0, 0, 0};
    uint32_t mn[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    uint32_t mx[4] = {0u, 0u, 0u, 0u};
    for (int b0 = 0; b0 < ((r1 - r0) << g.shift); b0 += TB) {
        float4 v[TB];
        bool on[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int blk = b0 + j;
            const int sg = r0 + (blk >> g.shift);
            on[j] = sg < r1 && uint64_t(sm.segkey[sg]) >= lo;
            v[j] = on[j] ? load4<VEC, NC>(row, g.V, g.base(sg, blk & mask, lane), fill)
                         : make_float4(fill, fill, fill, fill);
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            if (!on[j]) continue;
            const int blk = b0 + j;
            const int base = g.base(r0 + (blk >> g.shift), blk & mask, lane);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xv = q_at(v[j], q);
                const uint32_t key = keyf(xv);
                const bool inr = base + q < g.V;
                const bool g0 = inr && key >= p0, g1 = inr && key >= p1, g2 = inr && key >= p2;
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
        }
    }
    // warp -> block (fixed order) -> the leader's part[rank]
    float* rf = reinterpret_cast<float*>(sm.red);
    uint32_t* ru = reinterpret_cast<uint32_t*>(sm.red);
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
            rf[i * NW + warp] = m[i];
            ru[(3 + i) * NW + warp] = uint32_t(c[i]);
        }
    }
    __syncthreads();
    uint32_t rec[6];
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) {
            float a = 0.f;
            uint32_t b = 0;
            for (int w = 0; w < NW; ++w) {
                a += rf[i * NW + w];
                b += ru[(3 + i) * NW + w];
            }
            rec[i] = __float_as_uint(a);
            rec[3 + i] = b;
        }
    }
    __syncthreads();
    if (lane == 0) {
        for (int t = 0; t < 4; ++t) {
            ru[t * NW + warp] = mn[t];
            ru[(4 + t) * NW + warp] = mx[t];
        }
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part[rank]);
        for (int t = 0; t < 4; ++t) {
            uint32_t a = 0xffffffffu, b = 0u;
            for (int w = 0; w < NW; ++w) {
                a = min(a, ru[t * NW + w]);
                b = max(b, ru[(4 + t) * NW + w]);
            }
            put_leader(dst + 4 + 3 + t, a, leader);   // u[3 + t]
            put_leader(dst + 4 + 7 + t, b, leader);   // u[7 + t]
        }
        for (int i = 0; i < 3; ++i) {
            put_leader(dst + i, rec[i], leader);          // f[i]
            put_leader(dst + 4 + i, rec[3 + i], leader);  // u[i]
        }
    }
}

// Count and mass (x > 0) of key >= t over this CTA's segments; the record goes to the
// leader's part[rank] (f[0] mass, u[0] count).  Block-collective.
template <bool VEC, bool NC, typename KEYF>
FS_NOINLINE __device__ void massge_pass(const float* __restrict__ row, const Geom& g, const Smem& sm, bool leader,
                                        int rank, uint32_t t, KEYF keyf, int warp, int lane, int tid) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const int mask = g.seg_it() - 1;
    float ms = 0.f;
    int cnt = 0;
    for (int blk = 0; blk < ((r1 - r0) << g.shift); ++blk) {
        const int sg = r0 + (blk >> g.shift);
        if (sm.segkey[sg] < t) continue;
        const int base = g.base(sg, blk & mask, lane);
        const float4 v = load4<VEC, NC>(row, g.V, base, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float xv = q_at(v, q);
            const bool gq = keyf(xv) >= t && xv > 0.f && base + q < g.V;
            ms += gq ? xv : 0.f;
            cnt += gq;
        }
    }
    ms = warp_sum(ms);
    cnt = warp_sum_i(cnt);
    float* rf = reinterpret_cast<float*>(sm.red);
    if (lane == 0) {
        rf[warp] = ms;
        sm.red[NW + warp] = cnt;
    }
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        int n = 0;
        for (int w = 0; w < NW; ++w) {
            a += rf[w];
            n += sm.red[NW + w];
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.part[rank]);
        put_leader(dst, __float_as_uint(a), leader);
        put_leader(dst + 4, uint32_t(n), leader);
    }
}

// Leader: one bisection step after all parts are in.  Updates the interval; returns
// nothing (the state is replicated in the caller's registers on the leader only).
struct Bisect {
    uint64_t lo, hi;   // crit(lo) holds, crit(hi) does not; done when hi = lo + 1
    float mass_lo;     // mass(key >= lo) (probabilities)
};

// Pivots of the next pass: three points splitting [lo, hi) into quarters (fewer when
// the interval is short; unused pivots equal hi).
__device__ __forceinline__ void bisect_pivots(const Bisect& st, uint32_t* piv) {
    const uint64_t d = st.hi - st.lo;
    if (d >= 4) {
#pragma unroll
        for (int i = 0; i < 3; ++i) piv[i] = uint32_t(st.lo + (d * uint64_t(i + 1)) / 4);
    } else {
        piv[0] = uint32_t(st.lo + 1);
        piv[1] = uint32_t(d == 3 ? st.lo + 2 : st.hi);
        piv[2] = uint32_t(st.hi);
    }
}

// Fold the C parts of a bisection pass into the interval ([drill] section 5: take the
// largest pivot where the criterion holds; shrink to the keys present).
template <bool MASS>
__device__ __forceinline__ void bisect_update(const Smem& sm, int C, Bisect& st, const uint32_t* piv, int kcrit,
                                              float target) {
    float mass[3] = {0.f, 0.f, 0.f};
    int cnt[3] = {0, 0, 0};
    uint32_t kmin[4], kmax[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        kmin[t] = 0xffffffffu;
        kmax[t] = 0u;
    }
    for (int c = 0; c < C; ++c) {
        const Part& p = sm.part[c];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            mass[i] += p.f[i];
            cnt[i] += int(p.u[i]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            kmin[t] = min(kmin[t], p.u[3 + t]);
            kmax[t] = max(kmax[t], p.u[7 + t]);
        }
    }
    int best = -1;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        if (uint64_t(piv[i]) < st.hi) {
            const bool ok = MASS ? (mass[i] >= target) : (cnt[i] >= kcrit);
            if (ok) best = i;
        }
    }
    uint64_t nlo = st.lo, nhi = st.hi;
    int bkt = 0;
    if (best >= 0) {
        nlo = piv[best];
        st.mass_lo = mass[best];
        bkt = best + 1;
    }
    if (best + 1 < 3 && uint64_t(piv[best + 1]) < st.hi) nhi = piv[best + 1];
    if (kmin[bkt] <= kmax[bkt]) {  // keys present in the new interval
        nlo = max(nlo, uint64_t(kmin[bkt]));
        nhi = min(nhi, uint64_t(kmax[bkt]) + 1);
    }
    st.lo = nlo;
    st.hi = nhi;
}

// Leader: drive a bisection to the end with the whole cluster (at most 40 passes).
template <bool VEC, bool NC, bool MASS, typename KEYF>
FS_NOINLINE __device__ void bisect_leader(const float* __restrict__ row, const Geom& g, const Smem& sm, int C,
                                          Bisect* stp, int kcrit, float target, KEYF keyf, float fill, int warp,
                                          int lane, int tid) {
    Bisect st = *stp;
    for (int iter = 0; iter < 40 && st.hi - st.lo > 1; ++iter) {
        uint32_t piv[3];
        bisect_pivots(st, piv);
        Ctl c{};
        c.cmd = CMD_BISECT;
        c.u[0] = piv[0];
        c.u[1] = piv[1];
        c.u[2] = piv[2];
        c.u[3] = uint32_t(st.lo);
        c.hi_lo = uint32_t(st.hi);
        c.hi_hi = uint32_t(st.hi >> 32);
        send_command(sm, c, C, tid);
        bisect_pass<VEC, NC, MASS>(row, g, sm, true, 0, st.lo, st.hi, piv, keyf, fill, warp, lane, tid);
        cluster_sync();  // every part is in
        bisect_update<MASS>(sm, C, st, piv, kcrit, target);
        __syncthreads();
    }
    *stp = st;
}

// Leader: count and mass of key >= t over the whole row, with the cluster.
template <bool VEC, bool NC, typename KEYF>
FS_NOINLINE __device__ void massge_leader(const float* __restrict__ row, const Geom& g, const Smem& sm, int C,
                                          uint32_t t, KEYF keyf, int warp, int lane, int tid, float* mass_out,
                                          int* cnt_out) {
    Ctl c{};
    c.cmd = CMD_MASSGE;
    c.u[0] = t;
    send_command(sm, c, C, tid);
    massge_pass<VEC, NC>(row, g, sm, true, 0, t, keyf, warp, lane, tid);
    cluster_sync();
    float m = 0.f;
    int n = 0;
    for (int r = 0; r < C; ++r) {
        m += sm.part[r].f[0];
        n += int(sm.part[r].u[0]);
    }
    __syncthreads();
    *mass_out = m;
    *cnt_out = n;
}

}  // namespace fsd
