// Filter-only kernels (sm_103a): top_k_renorm_probs, top_p_renorm_probs,
// top_k_mask_logits.
//
// Each finds the exact threshold t on the integer order key of the row's values
// ([drill] sections 2-4: the largest t with count(key >= t) >= k, or with
// mass(key >= t) >= top_p * M), then writes the row once.  One cluster per row:
//   pass 1   one HBM read: per-segment maximum key, the row total and a bad flag;
//   search   top-k: a lower bound of t from a histogram of the segment maxima (the
//            k-th largest of any subset of the row is at most the row's), every CTA's
//            elements at or above it gathered into rank 0's list, and t counted
//            exactly among them; a bisection on the key takes over when they do not
//            fit on chip.
//            top-p: a histogram of integer masses over the key's top 11 bits picks
//            the bin where the prefix mass crosses top_p * M, the elements of that
//            bin are gathered to rank 0, which finishes with two radix rounds over
//            them (topp_threshold);
//   write    keep key >= t (x / kept mass, or the logit), else 0 / -inf.  Segments
//            whose maximum is below t are written without being read.
#include <type_traits>

#include "fs_device.cuh"
#include "fs_host.h"

namespace fsd {

enum { K_TOPK = 0, K_TOPP = 1, K_MASK = 2 };

struct FilterArgs {
    const float* in;
    float* out;
    int V;
    const int* top_k;
    const float* top_p;
    unsigned char* out_valid;
    int shift;
    int ns;
    int nsc;
};

// Write `fill` over this CTA's segments whose largest key is below `floor`: their
// output is fill whatever the threshold, as long as it is at least `floor`.  No
// reads; streaming stores (the zeros are not read again).
template <bool VEC>
__device__ __forceinline__ void fill_below(float* __restrict__ orow, Geom g, Smem sm, uint32_t floor, float fill,
                                           int warp, int lane) {
    int r0, r1;
    warp_range(g.s1 - g.s0, warp, r0, r1);
    r0 += g.s0;
    r1 += g.s0;
    const bool vec_out = VEC && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
#pragma unroll 1
    for (int sg = r0; sg < r1; ++sg) {
        if (sm.segkey()[sg] >= floor) continue;
#pragma unroll 1
        for (int it = 0; it < g.seg_it(); ++it) {
            const int base = g.base(sg, it, lane);
            if (vec_out && base + 3 < g.V) {
                __stcs(reinterpret_cast<float4*>(orow + base), make_float4(fill, fill, fill, fill));
            } else {
#pragma unroll 1
                for (int q = 0; q < 4; ++q)
                    if (base + q < g.V) __stcs(orow + base + q, fill);
            }
        }
    }
}

// Write this CTA's segments: keep key >= t (x / denom, or the logit), else fill.
// Segments whose maximum key is below t are written without being read; those below
// `floor` were written already (fill_below) and are skipped.
template <bool VEC, int KIND>
__device__ __forceinline__ void write_pass(const float* __restrict__ row, float* __restrict__ orow, Geom g,
                                       Smem sm, bool valid, uint32_t t, float denom, int warp, int lane,
                                       uint32_t floor = 0u) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyLogit, KeyProb>::type;
    constexpr bool IS_PROB = KIND != K_MASK;
    const KEYF keyf;
    const float fill = IS_PROB ? 0.f : __int_as_float(0xff800000);
    const bool vec_out = VEC && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
    stream_warp<VEC, false>(
        row, g, sm, warp, lane, [&](int sg) { return valid && sm.segkey()[sg] >= t; },
        [&](int sg, int, bool on, const float4& v, int base) {
            if (sm.segkey()[sg] < floor) return;
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xv = q_at(v, q);
                o[q] = (on && keyf(xv) >= t) ? (IS_PROB ? xv / denom : xv) : fill;
            }
            if (vec_out && base + 3 < g.V) {
                *reinterpret_cast<float4*>(orow + base) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll 1
                for (int q = 0; q < 4; ++q)
                    if (base + q < g.V) orow[base + q] = o[q];
            }
        });
}

// The other CTAs: follow the leader's commands until the write.
template <bool VEC, int KIND>
__device__ __forceinline__ void filter_peer(const float* __restrict__ row, float* __restrict__ orow, Geom g,
                                            Smem sm, int rank, int C, int warp, int lane, int tid) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyLogit, KeyProb>::type;
    constexpr bool IS_PROB = KIND != K_MASK;
    for (;;) {
        cluster_sync();  // the command is published
        const Ctl c = *sm.ctl();
        const uint64_t hi = uint64_t(c.hi_lo) | (uint64_t(c.hi_hi) << 32);
        if (c.cmd == CMD_SEARCH) {
            search_pass<VEC, false, IS_PROB>(row, g, sm, false, rank, c.u[0], hi, KEYF(), warp, lane, tid);
        } else if (c.cmd == CMD_COLLECT) {
            collect_own<VEC>(row, g, sm, false, rank, C, rank * (CAP / C), CAP / C, c.u[0], hi, KEYF(), false, true,
                             warp, lane, tid);
        } else if (c.cmd == CMD_WRITE) {
            write_pass<VEC, KIND>(row, orow, g, sm, c.flag != 0, c.u[0], c.f[0], warp, lane);
            return;
        } else {
            return;  // CMD_EXIT
        }
        cluster_sync();  // the results are in the leader
        if (c.cmd == CMD_COLLECT) settle_list<VEC>(row, g, sm, false, rank, C, c.u[0], hi, KEYF(), false, warp, lane, tid);
    }
}

// Add the non-zero words of the local histogram L[0, nb) into every CTA's copy of R.
__device__ __forceinline__ void push_bins_u64(const unsigned long long* L, unsigned long long* R, int nb, int rank,
                                              int C, int tid) {
#pragma unroll 1
    for (int bin = tid; bin < nb; bin += NT) {
        const unsigned long long v = L[bin];
        if (!v) continue;
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
            if (r == rank) {
                atomicAdd(&R[bin], v);
            } else {
                asm volatile("red.shared::cluster.add.u64 [%0], %1;" ::"r"(map_rank(smem_u32(&R[bin]), uint32_t(r))),
                             "l"(v)
                             : "memory");
            }
        }
    }
}

// Add the 32-bit words of the local histogram L[0, nb) into every CTA's copy of R.
__device__ __forceinline__ void push_bins_u32(const uint32_t* L, uint32_t* R, int nb, int rank, int C, int tid) {
#pragma unroll 1
    for (int bin = tid; bin < nb; bin += NT) {
        const uint32_t v = L[bin];
        if (!v) continue;
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
            if (r == rank) {
                atomicAdd(&R[bin], v);
            } else {
                asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(map_rank(smem_u32(&R[bin]), uint32_t(r))),
                             "r"(v)
                             : "memory");
            }
        }
    }
}

constexpr int TOPP_LIST = 2048;  // entries of the leader's list of crossing-bin elements

// Exact 64-bit histogram passes over the keys of the window [lo, hi), narrowing it to
// the key where the prefix mass from the top reaches the target: the fallback of
// topp_threshold when the crossing bin holds more elements than the leader's list.
// Masses x * 2^sh are rounded to integers, with the row maximum below 2^42 (the row's
// sum stays below 2^63); the first pass also sums, in registers, the row total (the
// target is ceil(top_p * total)) and the mass above the window.  Each pass keeps the
// bin where the prefix reaches the target, until a bin is one key wide.  Block- and
// cluster-collective; both receive buffers are zero on entry and no CTA adds to them
// before the cluster barrier that precedes the call.
template <bool VEC>
__device__ __forceinline__ void topp_exact_levels(const float* __restrict__ row, Geom g, Smem sm, int rank, int C,
                                                  uint32_t maxkey, float tp, unsigned long long lo,
                                                  unsigned long long hi, int warp, int lane, int tid, uint32_t& t_out,
                                                  float& denom_out) {
    using u64 = unsigned long long;
    constexpr int TW = int(Layout::TOPPW);
    u64* L = sm.topp_local();
    u64* b64 = reinterpret_cast<u64*>(sm.red() + 64);  // [6] broadcast words
    const int sh = 168 - int((maxkey >> 23) & 255u);     // the maximum * 2^sh < 2^42
    u64 A = 0, T = 1;  // the mass above the window, the target
    uint32_t t = uint32_t(lo);
    u64 kept = 0;
#pragma unroll 1
    for (int lev = 0; lev < 4; ++lev) {
        const bool first = lev == 0;
        int lw = 0;
        while (((hi - lo + (1ull << lw) - 1) >> lw) > u64(HBINS)) ++lw;
        const int nb = int((hi - lo + (1ull << lw) - 1) >> lw);
        u64* R = sm.topp_recv(lev & 1);
        for (int i = tid; i < TW; i += NT) L[i] = 0ull;
        __syncthreads();
        u64 a_above = 0, a_total = 0;
        const uint32_t live_lo = first ? 1u : uint32_t(lo);
        stream_warp<VEC, true>(
            row, g, sm, warp, lane, [&](int sg) { return sm.segkey()[sg] >= live_lo; },
            [&](int, int, bool on, const float4& v, int) {
                if (!on) return;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x = q_at(v, q);
                    const u64 key = prob_key(x);
                    if (first) {
                        const u64 m = fixed_point(x, sh);
                        a_total += m;
                        if (key >= hi) a_above += m;
                    }
                    if (key >= lo && key < hi) atomicAdd(&L[(key - lo) >> lw], fixed_point(x, sh));
                }
            });
        if (first) {
            a_above = warp_sum_u64(a_above);
            a_total = warp_sum_u64(a_total);
            if (lane == 0) {
                atomicAdd(&L[HBINS], a_above);
                atomicAdd(&L[HBINS + 1], a_total);
            }
        }
        __syncthreads();
        push_bins_u64(L, R, nb, rank, C, tid);
        if (first) push_bins_u64(L + HBINS, R + HBINS, 2, rank, C, tid);
        if (lev >= 1)  // the other buffer, for the next pass: read before this pass began
            for (int i = tid; i < TW; i += NT) sm.topp_recv((lev + 1) & 1)[i] = 0ull;
        cluster_sync();  // this pass's sums in every R
        if (warp == 0) {
            if (first) {
                const u64 total = R[HBINS + 1];
                A = R[HBINS];
                if (tp > 0.f) {
                    const double tt = ceil(double(tp) * double(total));
                    T = tt < 1.0 ? 1ull : u64(tt);
                }
            }
            const int top = int(min(u64(nb - 1), (u64(maxkey) - lo) >> lw));
            u64 above;
            const int j = max(0, scan_bins_down<u64>(R, top, T > A ? T - A : 1ull, lane, above));
            if (lane == 0) {
                const u64 nlo = lo + (u64(j) << lw);
                b64[0] = nlo;
                b64[1] = min(hi, nlo + (1ull << lw));
                b64[2] = A + above;
                b64[3] = T;
                b64[4] = A + above + R[j];
                b64[5] = lw == 0 ? 1ull : 0ull;
            }
        }
        __syncthreads();
        lo = b64[0];
        hi = b64[1];
        A = b64[2];
        T = b64[3];
        t = uint32_t(lo);
        kept = b64[4];
        if (b64[5]) break;
        __syncthreads();  // b64 is rewritten by the next pass
    }
    t_out = t;
    denom_out = float(double(kept) * ldexp(1.0, -sh));
}

// Block- and cluster-collective top-p threshold of a valid row of probabilities: the
// largest key t with mass(key >= t) >= top_p * M ([drill] section 4; top_p <= 0 keeps
// the maximum alone).  Returns t and the kept mass, the same in every CTA.
//   level 0   every CTA counts its share of the row (which pass 1 left in L2) into
//             bins of key bits 31..21 with 32-bit masses x * 2^s rounded to integers
//             (M * 2^s < 2^31, so no sum overflows; integer sums do not depend on the
//             order of the additions) and adds them into every CTA's copy; every CTA
//             then picks the bin B where the prefix mass from the top reaches
//             top_p times the row's sum of those masses.
//   collect   every CTA sums (fp32, in its own fixed order) its elements above B and
//             appends the elements inside B, as (key, x * 2^sh rounded, the maximum *
//             2^sh < 2^42), to the leader's list (slots reserved per warp with one
//             cluster-shared atomic).
//   finish    the leader: the mass above B (the CTAs' sums added in rank order) and
//             the target top_p * M, in units of 2^-sh, then two radix rounds over the
//             list (key bits 20..10, then 9..0) with 64-bit mass histograms; the
//             result goes to every CTA before one cluster barrier.  If rounding put
//             the target outside B's range of masses, the crossing is at B's edge:
//             t = the key above B (the target was reached there) or B's lowest key.
// When B holds more elements than the list, every CTA runs topp_exact_levels on B.
// The receive buffers are zero on entry (cleared before the cluster barrier after
// pass 1), and so is the leader's list count, red[100].
template <bool VEC>
__device__ __forceinline__ void topp_threshold(const float* __restrict__ row, Geom g, Smem sm, bool leader, int rank,
                                               int C, uint32_t maxkey, float M, float tp, int warp, int lane, int tid,
                                               uint32_t& t_out, float& denom_out) {
    using u64 = unsigned long long;
    constexpr int TW = int(Layout::TOPPW);
    u64* L = sm.topp_local();
    u64* b64 = reinterpret_cast<u64*>(sm.red() + 64);  // [6] broadcast words
    uint32_t* list_n = reinterpret_cast<uint32_t*>(sm.red() + 100);
    u64* list_q = sm.topp_recv(0);                                                      // [TOPP_LIST] masses
    uint32_t* list_k = reinterpret_cast<uint32_t*>(sm.topp_recv(1)) + HBINS;            // [TOPP_LIST] keys
    uint32_t* R32 = reinterpret_cast<uint32_t*>(sm.topp_recv(1));                       // [HBINS] level 0
    // ---- level 0
    {
        const int s0 = 157 - int(__float_as_uint(M) >> 23);  // M * 2^s0 < 2^31
        const int s0a = s0 > 126 ? 126 : s0;
        const float f0a = __int_as_float((s0a + 127) << 23), f0b = __int_as_float((s0 - s0a + 127) << 23);
        uint32_t* L32 = reinterpret_cast<uint32_t*>(L);
        for (int i = tid; i < HBINS; i += NT) L32[i] = 0u;
        __syncthreads();
        stream_warp<VEC, true>(
            row, g, sm, warp, lane, [&](int sg) { return sm.segkey()[sg] != 0u; },
            [&](int, int, bool on, const float4& v, int) {
                if (!on) return;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x = q_at(v, q);
                    if (x > 0.f) atomicAdd(&L32[__float_as_uint(x) >> 21], __float2uint_rn((x * f0a) * f0b));
                }
            });
        __syncthreads();
        push_bins_u32(L32, R32, HBINS, rank, C, tid);
        cluster_sync();  // level-0 sums in every R32
        if (warp == 0) {
            u64 q = 0;
            for (int i = lane; i < HBINS; i += 32) q += R32[i];
            q = warp_sum_u64(q);
            const double T0 = tp > 0.f ? ceil(double(tp) * double(q)) : 1.0;
            uint32_t ab;
            const int B = scan_bins_down<uint32_t>(R32, int(maxkey >> 21), uint32_t(T0 < 1.0 ? 1.0 : T0), lane, ab);
            if (lane == 0) b64[0] = u64(max(B, 0));
        }
        __syncthreads();
    }
    const uint32_t B = uint32_t(b64[0]);
    const uint32_t lo = B << 21;
    const u64 hi = u64(B + 1) << 21;
    const int sh = 168 - int((maxkey >> 23) & 255u);
    // ---- collect
    float a_f = 0.f;
    const uint32_t cnt_addr = map_rank(smem_u32(list_n), 0);
    stream_warp<VEC, true>(
        row, g, sm, warp, lane, [&](int sg) { return sm.segkey()[sg] >= lo; },
        [&](int, int, bool on, const float4& v, int) {
            if (!on) return;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = q_at(v, q);
                const uint32_t key = prob_key(x);
                if (key >= hi) a_f += x;
                const bool in = key >= lo && u64(key) < hi;
                const unsigned bal = __ballot_sync(FULL, in);
                if (bal) {
                    uint32_t base = 0;
                    if (lane == 0)  // the same cluster-scoped atomic in every CTA, the leader included
                        asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;"
                                     : "=r"(base)
                                     : "r"(cnt_addr), "r"(uint32_t(__popc(bal)))
                                     : "memory");
                    base = __shfl_sync(FULL, base, 0);
                    const uint32_t pos = base + uint32_t(__popc(bal & ((1u << lane) - 1u)));
                    if (in && pos < uint32_t(TOPP_LIST)) {
                        const u64 m = fixed_point(x, sh);
                        if (leader) {
                            list_k[pos] = key;
                            list_q[pos] = m;
                        } else {
                            st_dsmem_u32(map_rank(smem_u32(&list_k[pos]), 0), key);
                            asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(map_rank(smem_u32(&list_q[pos]), 0)),
                                         "l"(m)
                                         : "memory");
                        }
                    }
                }
            }
        });
    a_f = warp_sum(a_f);
    if (lane == 0) reinterpret_cast<float*>(sm.red())[warp] = a_f;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += reinterpret_cast<float*>(sm.red())[w];
        put_leader(&sm.part()[rank].f[3], __float_as_uint(s), leader);
    }
    cluster_sync();  // the list, its count and the CTAs' sums are in the leader
    uint32_t n_all;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(n_all) : "r"(cnt_addr) : "memory");
    if (n_all > uint32_t(TOPP_LIST)) {  // the fallback, in every CTA alike
        cluster_sync();                  // every CTA has read the count
        for (int i = tid; i < 2 * TW; i += NT) sm.topp_recv(0)[i] = 0ull;
        cluster_sync();                  // every receive buffer is clear
        topp_exact_levels<VEC>(row, g, sm, rank, C, maxkey, tp, lo, hi, warp, lane, tid, t_out, denom_out);
        return;
    }
    // ---- finish (leader)
    if (leader) {
        const int n = int(n_all);
        if (tid == 0) {
            float af = 0.f;
            for (int r = 0; r < C; ++r) af += sm.part()[r].f[3];
            const double sc = ldexp(1.0, sh);
            const u64 A = u64(rint(double(af) * sc));
            const double tt = tp > 0.f ? ceil(double(tp) * double(M) * sc) : 1.0;
            b64[0] = A;
            b64[1] = tt < 1.0 ? 1ull : u64(tt);
            reinterpret_cast<float*>(sm.red())[96] = af;
        }
        for (int i = tid; i < HBINS; i += NT) L[i] = 0ull;
        __syncthreads();
        const u64 A = b64[0], T = b64[1];
        for (int i = tid; i < n; i += NT) atomicAdd(&L[(list_k[i] >> 10) & (HBINS - 1)], list_q[i]);
        __syncthreads();
        // round 1: bits 20..10
        if (warp == 0) {
            u64 w = 0;
            for (int i = lane; i < HBINS; i += 32) w += L[i];
            w = warp_sum_u64(w);
            int d1 = -1;  // -1: the target is reached above B; -2: only below B's lowest key
            u64 ab = 0;
            if (T > A && T <= A + w) {
                const int top = (maxkey >> 21) == B ? int((maxkey >> 10) & (HBINS - 1)) : HBINS - 1;
                d1 = max(0, scan_bins_down<u64>(L, top, T - A, lane, ab));
            } else if (T > A) {
                d1 = -2;
            }
            if (lane == 0) {
                b64[2] = u64(int64_t(d1));
                b64[3] = ab;
                b64[4] = w;
            }
        }
        __syncthreads();
        const int d1 = int(int64_t(b64[2]));
        uint32_t t;
        u64 kept_in;  // mass of the list at or above t
        if (d1 >= 0) {
            const uint32_t pre = (B << 11) | uint32_t(d1);
            const u64 ab1 = b64[3];
            for (int i = tid; i < 1024; i += NT) L[HBINS - 1024 + i] = 0ull;  // round-2 bins after round 1's
            __syncthreads();
            u64* L2 = L + (HBINS - 1024);
            for (int i = tid; i < n; i += NT)
                if ((list_k[i] >> 10) == pre) atomicAdd(&L2[list_k[i] & 1023u], list_q[i]);
            __syncthreads();
            if (warp == 0) {
                const int top = (maxkey >> 10) == pre ? int(maxkey & 1023u) : 1023;
                u64 ab2;
                const int d2 = max(0, scan_bins_down<u64>(L2, top, T - A - ab1, lane, ab2));
                if (lane == 0) {
                    b64[5] = u64(d2);
                    b64[3] = ab1 + ab2 + L2[d2];
                }
            }
            __syncthreads();
            t = (pre << 10) | uint32_t(b64[5]);
            kept_in = b64[3];
        } else if (d1 == -1) {
            t = uint32_t(min(hi, u64(0xffffffffu)));  // keep what lies above B
            kept_in = 0;
        } else {
            t = lo;  // keep all of B
            kept_in = b64[4];
        }
        if (tid == 0) {
            const float af = reinterpret_cast<float*>(sm.red())[96];
            const float denom = af + float(double(kept_in) * ldexp(1.0, -sh));
            for (int r = 0; r < C; ++r) {  // into every CTA's own slot
                if (r == 0) {
                    sm.part()[0].u[8] = t;
                    sm.part()[0].u[9] = __float_as_uint(denom);
                } else {
                    st_dsmem_u32(map_rank(smem_u32(&sm.part()[r].u[8]), uint32_t(r)), t);
                    st_dsmem_u32(map_rank(smem_u32(&sm.part()[r].u[9]), uint32_t(r)), __float_as_uint(denom));
                }
            }
        }
    }
    cluster_sync();  // t and the kept mass are in every CTA
    t_out = sm.part()[rank].u[8];
    denom_out = __uint_as_float(sm.part()[rank].u[9]);
}

// The single-pass kinds run at most 3 CTAs per SM (the launch plan's cap), so they are
// compiled for 3 and keep their working set in registers; top-p renorm takes the
// occupancy limit for its multi-pass plan.
template <bool VEC, int KIND>
__global__ void __launch_bounds__(NT, KIND == K_TOPP ? 4 : 3) filter_kernel(const FilterArgs a) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyLogit, KeyProb>::type;
    constexpr bool IS_PROB = KIND != K_MASK;
    const KEYF keyf;
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool leader = rank == 0;
    const Smem sm(a.ns);
    const Geom g(a.V, a.shift, a.ns, a.nsc, rank);
    const int V = a.V, ns = a.ns;
    grid_dependency_wait();
    allow_dependents();
    const float* row = a.in + size_t(b) * size_t(V);
    float* orow = a.out + size_t(b) * size_t(V);

    const int k = (KIND != K_TOPP) ? a.top_k[b] : 0;
    const float tp = (KIND == K_TOPP) ? a.top_p[b] : 1.f;
    const bool k_on = KIND != K_TOPP && k > 0 && k < V;
    const bool need_hist = k_on && ns >= k;

    // ---- pass 1, inside a split cluster barrier
    if (need_hist)
        for (int i = tid; i < HBINS; i += NT) {
            sm.hist()[i] = 0u;
            sm.hist()[HBINS + i] = 0u;
            reinterpret_cast<uint32_t*>(sm.lv())[i] = 0u;
        }
    if (tid == 0) *sm.ctr() = NW;
    __syncthreads();
    cluster_arrive();
    int pos = 0;
    bool bad = false;
    uint32_t kmax = 0;
    pass1<VEC, false, IS_PROB>(row, g, sm, need_hist ? 21 : -1, warp, lane, pos, bad,
                               kmax);
    cluster_wait();  // every CTA has started and cleared its histogram
    pass1_totals(g, sm, leader, rank, C, pos, bad, kmax, need_hist ? 21 : -1, IS_PROB, false, warp,
                 lane, tid, false, need_hist ? k : 0);
    if (KIND == K_TOPP) {  // the top-p receive buffers (over the segment masses, now read) and list count
        for (int i = tid; i < 2 * int(Layout::TOPPW); i += NT) sm.topp_recv(0)[i] = 0ull;
        if (tid == 0) sm.red()[100] = 0;
    }
    cluster_sync();  // every CTA's parts and histogram are complete

    const Totals tot = cluster_totals(sm, C);
    const bool any_bad = tot.any_bad;
    const float M = tot.M;
    const uint32_t maxkey = tot.maxkey;
    bool valid = !any_bad;
    if (IS_PROB) valid = valid && M > 0.f && M <= 3.402823466e38f;
    if (KIND == K_TOPP && isnan(tp)) valid = false;

    // ---- top-k: every CTA derives the same lower bound L0 <= t from its copy of the
    // histogram and sends its elements >= L0 to its region of every CTA's list.  When
    // the list is complete, each CTA finds t and the kept mass itself and writes its
    // share.
    uint32_t L0 = 0u;
    int list_mode = -1;  // 0: regions fit, 1: contiguous, -1: no list
    const bool early = valid && need_hist && orow != row;  // fill the sure part of the output early
    if (k_on) {
        L0 = need_hist ? hist_bound(sm, g, rank, C, k, maxkey, warp, lane, tid) : 0u;
        if (IS_PROB) L0 = max(L0, 1u);
        collect_own<VEC>(row, g, sm, leader, rank, C, rank * (CAP / C), CAP / C, L0, NO_LIMIT, keyf, true, true,
                         warp, lane, tid);
        // While the other CTAs finish their candidates: the output of the segments whose
        // maximum is below L0 (<= t) is the fill, written now when it does not alias the
        // input (an in-place call keeps the row intact for the fallback search).
        cluster_arrive();
        if (early) fill_below<VEC>(orow, g, sm, L0, IS_PROB ? 0.f : __int_as_float(0xff800000), warp, lane);
        cluster_wait();  // every region and count is in every CTA
        list_mode = settle_list<VEC>(row, g, sm, leader, rank, C, L0, NO_LIMIT, keyf, true, warp, lane, tid);
    }
    if (list_mode >= 0) {
        // Every element >= L0 (hence >= t) is in the list.
        const int n = regions_total(sm, C);
        if (n <= SMALL) {  // the usual case: in warp 0's registers
            if (warp == 0) {
                const Small sl = small_gather(sm, C, CAP / C, list_mode == 1, lane);
                const uint32_t t = small_kth(sl, k, keyf);
                float s = 0.f;
#pragma unroll
                for (int r = 0; r < SR; ++r) s += sl.in[r] && keyf(sl.x[r]) >= t ? sl.x[r] : 0.f;
                s = warp_sum(s);
                if (lane == 0) {
                    sm.red()[40] = int(t);
                    reinterpret_cast<float*>(sm.red())[41] = s;
                }
            }
        } else {  // a longer list: joined, then a radix select by the whole CTA
            if (list_mode == 0 && warp == 0) join_regions_warp(sm, C, CAP / C, lane);
            __syncthreads();
            const uint32_t t = kth_key_cta(sm, n, k, keyf, warp, lane, tid);
            if (warp == 0) {
                float s = 0.f;
                for (int i = lane; i < n; i += 32) s += keyf(sm.lv()[i]) >= t ? sm.lv()[i] : 0.f;
                s = warp_sum(s);
                if (lane == 0) {
                    sm.red()[40] = int(t);
                    reinterpret_cast<float*>(sm.red())[41] = s;
                }
            }
        }
        __syncthreads();
        const uint32_t t = uint32_t(sm.red()[40]);
        const float denom = reinterpret_cast<float*>(sm.red())[41];
        write_pass<VEC, KIND>(row, orow, g, sm, valid, t, denom, warp, lane, early ? L0 : 0u);
        if (leader && tid == 0 && a.out_valid) a.out_valid[b] = valid ? 1 : 0;
        return;
    }
    if (KIND == K_TOPP) {  // every CTA alike: the threshold, then its share of the row
        uint32_t t = 0;   // keep key >= t
        float denom = M;  // kept mass
        if (valid && tp < 1.f) topp_threshold<VEC>(row, g, sm, leader, rank, C, maxkey, M, tp, warp, lane, tid, t, denom);
        write_pass<VEC, KIND>(row, orow, g, sm, valid, t, denom, warp, lane);
        if (leader && tid == 0 && a.out_valid) a.out_valid[b] = valid ? 1 : 0;
        return;
    }
    if (!leader) {
        filter_peer<VEC, KIND>(row, orow, g, sm, rank, C, warp, lane, tid);
        return;
    }

    // ---- leader: the threshold with the cluster's help, then everyone writes
    uint32_t t = 0;   // keep key >= t
    float denom = M;  // kept mass (probabilities)
    if (valid) {
        if (KIND != K_TOPP) {
            if (k_on) {
                // More than CAP candidates: the threshold by a search with the cluster.
                Search st = search_start(maxkey, M, V);
                threshold_search<VEC, false, false, IS_PROB>(row, g, sm, C, st, k, 0.f, keyf, warp, lane, tid);
                t = uint32_t(st.lo);
                denom = st.mass_lo;
            }
        }
    }

    // ---- everyone writes its share of the row
    Ctl c{};
    c.cmd = CMD_WRITE;
    c.flag = valid ? 1 : 0;
    c.u[0] = t;
    c.f[0] = denom;
    send_command(sm, c, C, tid);
    write_pass<VEC, KIND>(row, orow, g, sm, valid, t, denom, warp, lane);
    if (tid == 0 && a.out_valid) a.out_valid[b] = valid ? 1 : 0;
}

template <int KIND>
static fs_status launch_filter(const float* in, int32_t batch, int32_t vocab, const int32_t* top_k,
                               const float* top_p, float* out, uint8_t* out_valid, void* stream) {
    if (batch < 0) return FS_ERR_INVALID_ARG;
    if (batch == 0) return FS_OK;
    if (!in || !out) return FS_ERR_INVALID_ARG;
    if (KIND == K_TOPP ? !top_p : !top_k) return FS_ERR_INVALID_ARG;
    if (vocab < 1) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(in) & 15) == 0);
    const void* fn = vec ? reinterpret_cast<const void*>(filter_kernel<true, KIND>)
                         : reinterpret_cast<const void*>(filter_kernel<false, KIND>);
    Plan p;
    fs_status st = make_plan(batch, vocab, fn, KIND != K_TOPP, p, KIND == K_TOPP);
    if (st != FS_OK) return st;
    FilterArgs a;
    a.in = in;
    a.out = out;
    a.V = vocab;
    a.top_k = top_k;
    a.top_p = top_p;
    a.out_valid = out_valid;
    a.shift = p.shift;
    a.ns = p.ns;
    a.nsc = p.nsc;
    if (vec) return launch_cluster(filter_kernel<true, KIND>, p, batch, stream, a);
    return launch_cluster(filter_kernel<false, KIND>, p, batch, stream, a);
}

}  // namespace fsd

extern "C" {

fs_status fs_top_k_renorm_probs(const float* probs, int32_t batch, int32_t vocab, const int32_t* top_k,
                                float* out_probs, uint8_t* out_valid, void* stream) {
    return fsd::launch_filter<fsd::K_TOPK>(probs, batch, vocab, top_k, nullptr, out_probs, out_valid, stream);
}

fs_status fs_top_p_renorm_probs(const float* probs, int32_t batch, int32_t vocab, const float* top_p,
                                float* out_probs, uint8_t* out_valid, void* stream) {
    return fsd::launch_filter<fsd::K_TOPP>(probs, batch, vocab, nullptr, top_p, out_probs, out_valid, stream);
}

fs_status fs_top_k_mask_logits(const float* logits, int32_t batch, int32_t vocab, const int32_t* top_k,
                               float* out_logits, uint8_t* out_valid, void* stream) {
    return fsd::launch_filter<fsd::K_MASK>(logits, batch, vocab, top_k, nullptr, out_logits, out_valid, stream);
}

}  // extern "C"
