// Dual-pivot rejection sampler (sm_103a).
//
// Two execution models.  The top-k-first samplers, the joint order with a top-k or a
// min-p filter and sampling without filters, on rows of probabilities, run as a scan
// of every input row spread evenly over the GPU (scan_kernel, writing a small summary
// of each row) and one finishing launch (kfirst_kernel, kjoint_kernel: one CTA per
// output row; kdraw_kernel: one warp per output row); see the sections below.  The
// other samplers run on one thread-block cluster per output row (sample_kernel; see
// fs_device.cuh for its execution model), and so do the rows the lean finishes hand
// over (the cluster code with a cluster of one, after the scan).
// The cluster sampler's steps, in the order the pages give them:
//   pass 1   every CTA reads its share of the row once; the leader ends up with every
//            segment's maximum key and mass, each CTA's mass, the row total M, the
//            positive count and a NaN/negative flag;
//   prologue (top-k-first only) the exact k-th largest value t_k and
//            F_k = mass(x >= t_k) ([explainer] filter order): a lower bound of t_k from
//            a histogram of the segment maxima (the k-th largest of any subset of the
//            row is at most the row's), every CTA's elements at or above it gathered
//            into the leader's list, and t_k counted exactly among them;
//   rounds   ([blog] dual-pivot rejection sampling) draw j by inverse transform over
//            {p > low}, pivot1 = p_j, pivot2 = (pivot1 + high) / 2, one fused
//            reduction of (mass, count) above both pivots, then accept j, or
//            (low, high) <- (pivot1, pivot2), or low <- pivot2.
// While many tokens lie above `low`, a round's reduction runs on the whole cluster
// over the segments whose maximum exceeds pivot1 (read again through L2); once at most
// CAP tokens are left, the leader gathers them in index order and finishes alone on
// one warp.
// Rows of logits (the from-logits entry, temperature T) are read once as well: pass 1
// keeps logit keys and, where draws over the whole row need them, each segment's mass
// relative to its own largest logit (an online softmax); after the first barrier the
// row's maximum m is known and every later read sees the weights exp((z - m) / T).
#include <mutex>

#include "fs_device.cuh"
#include "fs_host.h"

namespace fsd {

struct SampleArgs {
    const float* probs;
    int batch_in;
    int V;
    const int* indices;
    const int* top_k;
    const float* top_p;
    const float* min_p;
    int order;                // 0 top_k_first, 1 joint
    unsigned long long seed, offset;
    const unsigned long long* seeds;       // per output row, nullable
    const unsigned long long* offsets;     // per output row, nullable
    const unsigned long long* offset_dev;  // added to every row's offset, nullable
    int single_pivot;         // 1: the one-pivot rule (ablation)
    const float* temperature; // rows of logits: per output row, nullable (1)
    int* out_token;
    unsigned char* out_valid;
    int* out_rounds;
    int shift;                // log2(blocks per segment)
    int ns;                   // segments per row
    int nsc;                  // segments per CTA
    // Finishing launch (FIN): the row summaries written by scan_kernel.
    const uint32_t* skey;     // [batch_in][ls] segment maxima (order keys)
    const float* smass;       // [batch_in][ls] segment masses (rows of probabilities)
    const uint4* sstat;       // [batch_in][nu] per unit: mass, 0, bad flag, largest key
    const uint32_t* scode;    // [batch_in][nu][32] run codes (SCAN_JOINT), nullable
    int ls;                   // words per row of skey / smass
    int nu;                   // units per row
    unsigned* sctr;           // the scan's claim counters, set back to zero by output row 0
    int nout;                 // output rows (kdraw_kernel: one warp per output row)
    // Joint-order finish (kjoint_kernel): 1 = the whole row is staged in shared memory;
    // 0 = candidate list, then a list of the elements above low of a.jy4 float4 runs.
    int jmode;
    int jy4;
};

// ------------------------------------------------------------------ row summaries
//
// The samplers that need nothing of a row after its one read but the top of it (the
// top-k-first order) or a single draw (no filter) run as two launches.  scan_kernel
// reads every input row once, spread evenly over the whole GPU: the unit of work is
// TB consecutive blocks of one row (a warp's trip, 2 KB), and warp w of the grid takes
// units w, w + W, w + 2W, ... of the matrix in row-major order (W warps in the grid),
// so every SM streams the same number of bytes whatever the batch.  Per unit it writes
// each segment's largest order key and mass, and the unit's mass, positive count, bad
// flag and largest key (no positive count: V bounds it).  The finishing launch
// (sample_kernel with FIN, one CTA per
// output row) reads the summary of its input row from L2 and goes on exactly as the
// one-CTA cluster does after pass 1.  Nothing in scan_kernel waits on another thread.
struct ScanArgs {
    const float* x;           // [rows][V]
    int rows, V, shift, ns, nu, ls;
    uint32_t* key;            // [rows][ls]
    float* mass;              // [rows][ls], rows of probabilities
    uint4* stat;              // [rows][nu]
    uint32_t* code;           // [rows][nu][32] SCAN_JOINT: lane l's word of unit q holds in byte j the code of
                              // run (q TB + j) 32 + l (the float4 of elements 4 times that)
    unsigned* ctr;            // claim counters of the last units, SCAN_CTR_STRIDE words apart (zero at launch)
    long long ustatic;        // units [0, ustatic) are dealt round-robin; the rest are claimed
    int slice;                // claimed units per counter
};

// The last fifth of the units is not dealt but claimed: warps that finish their share
// early (SMs that happen to stream faster) take more.  The claimed units are cut into
// SCAN_CTRS slices, each with its own counter, and warp w claims from slice w % SCAN_CTRS
// only (one atomic per claimed unit, one more when its slice is used up); the finishing
// launch sets the counters back to zero once the scan is complete.
constexpr int SCAN_CTRS = 16;
// The scratch layout: the counters first (at a fixed place whatever the shape, so that
// a buffer reused for another shape still finds them at zero), then the segment keys,
// the segment masses, the unit records and the run codes.
constexpr int SCAN_CTR_STRIDE = 32;  // words between counters: one 128-byte line each (different L2 slices)
constexpr size_t SCAN_HEAD = size_t(SCAN_CTRS) * SCAN_CTR_STRIDE * 4;

__host__ __device__ inline int scan_units(int V) { return (V + TB * BLK - 1) / (TB * BLK); }
__host__ __device__ inline int scan_row_words(int ns) { return (ns + 3) & ~3; }

size_t scan_workspace_bytes(int batch_in, int vocab, bool codes) {
    const int shift = seg_shift_for(vocab);
    const int ns = (vocab + (BLK << shift) - 1) / (BLK << shift);
    const size_t ls = size_t(scan_row_words(ns));
    return SCAN_HEAD + size_t(batch_in) * (2 * ls * 4 + size_t(scan_units(vocab)) * (16 + (codes ? 32 * 4 : 0)));
}

// Kinds of summary.  SCAN_KEYS (rows of probabilities, paths that draw only from
// gathered candidates): segment maxima and unit totals.  SCAN_MASSES: segment masses
// as well (a draw over the whole row).  SCAN_LOGITS: maxima as logit keys, no masses
// (they depend on the temperature).  SCAN_JOINT: SCAN_MASSES and a one-byte code of
// every float4 run, min(255, key of its largest value >> 22) (the binade and its top
// mantissa bit, saturated): a run with an element above x has a code at least x's, so
// a pass for the elements above x reads the codes and only the runs they admit.
enum : int { SCAN_KEYS = 0, SCAN_MASSES = 1, SCAN_LOGITS = 2, SCAN_JOINT = 3 };
__host__ __device__ inline uint32_t run_code(uint32_t key) { return min(255u, key >> 22); }

// Per lane and block of four values, a few min / max / add instructions: the block's
// largest value (its order key after the warp maximum), its smallest (a negative one
// marks the row bad) and its sum.  A NaN passes through the sums and makes the row's
// total NaN, which the finishing launch treats as invalid; for logits a NaN sum or a
// +inf maximum marks the unit bad.  The unit record: mass (sum of its values, in
// block order), 0, bad flag, largest key.
template <bool VEC, int KIND>
__global__ void __launch_bounds__(NT, 4) scan_kernel(const ScanArgs a) {
    grid_dependency_wait();
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const long long total = (long long)a.rows * a.nu;
    const long long step = (long long)gridDim.x * NW;
    const int spu = TB >> a.shift;  // segments per unit
    constexpr bool LOGITS = KIND == SCAN_LOGITS;
    constexpr bool MASSES = KIND == SCAN_MASSES || KIND == SCAN_JOINT;
    const float fill = LOGITS ? __int_as_float(0xff800000) : 0.f;
    auto load_unit = [&](long long u, float4* v) {
        if (u < total) {
            const int r = int(u / a.nu), q = int(u - (long long)r * a.nu);
            const float* row = a.x + size_t(r) * size_t(a.V);
#pragma unroll
            for (int j = 0; j < TB; ++j) v[j] = load4<VEC, true>(row, a.V, (q * TB + j) * BLK + lane * 4, fill);
        } else {
#pragma unroll
            for (int j = 0; j < TB; ++j) v[j] = make_float4(fill, fill, fill, fill);
        }
    };
    const long long gw = (long long)blockIdx.x * NW + (threadIdx.x >> 5);
    const int home = int(gw % SCAN_CTRS);  // the warps of one counter are spread over every SM
    // This warp's units: its dealt ones gw, gw + step, ... below ustatic, then claims.  A
    // claim's atomic is issued one unit ahead (lane 0) and read at the next call, so its
    // round trip overlaps the unit being streamed.  Warp-collective.
    long long s_next = gw;
    bool pending = false;
    unsigned pend = 0u;
    auto issue = [&]() {
        if (lane == 0) pend = atomicAdd(&a.ctr[home * SCAN_CTR_STRIDE], 1u);
        pending = true;
    };
    auto next_unit = [&]() -> long long {
        if (s_next < a.ustatic) {
            const long long r = s_next;
            s_next += step;
            if (s_next >= a.ustatic && !pending) issue();
            return r;
        }
        if (!pending) issue();
        const long long uu = a.ustatic + (long long)home * a.slice + pend;
        const long long r = __shfl_sync(FULL, (pend < unsigned(a.slice) && uu < total) ? uu : total, 0);
        pending = false;
        if (r < total) issue();
        return r;
    };
    long long u = next_unit();
    float4 A[TB], Bv[TB];
    load_unit(u, A);
#pragma unroll 1
    while (u < total) {
        const long long un = next_unit();
        load_unit(un, Bv);
        const int r = int(u / a.nu), q = int(u - (long long)r * a.nu);
        uint32_t km[TB];
        float s[TB];
        float lo = 0.f;
        bool bad = false;
        uint32_t cw = 0u;  // SCAN_JOINT: the lane's four run codes
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const float4 v = A[j];
            const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
            if (KIND == SCAN_JOINT) cw |= run_code(prob_key(mx)) << (8 * j);
            s[j] = (v.x + v.y) + (v.z + v.w);
            if (LOGITS) {
                bad |= isnan(s[j]) || mx == __int_as_float(0x7f800000);
                km[j] = __reduce_max_sync(FULL, logit_key(mx));
            } else {
                lo = fminf(lo, fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
                km[j] = __reduce_max_sync(FULL, prob_key(mx));
            }
        }
        if (!LOGITS) bad = lo < 0.f;
        float um = 0.f;
        if (KIND == SCAN_JOINT) a.code[(size_t(r) * a.nu + q) * 32 + lane] = cw;
        if (MASSES) {
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < TB; ++j) s[j] += __shfl_xor_sync(FULL, s[j], m);
#pragma unroll
            for (int j = 0; j < TB; ++j) um += s[j];
        } else if (KIND == SCAN_KEYS) {
#pragma unroll
            for (int j = 0; j < TB; ++j) um += s[j];
            um = warp_sum(um);
        }
        // Lane l < spu: segment q * spu + l, its blocks combined in order.
        const int sg = q * spu + lane;
        if (lane < spu && sg < a.ns) {
            float ss = 0.f;
            uint32_t kk = 0;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const bool mine = (j >> a.shift) == lane;
                ss += mine ? s[j] : 0.f;
                kk = mine ? max(kk, km[j]) : kk;
            }
            a.key[size_t(r) * a.ls + sg] = kk;
            if (MASSES) a.mass[size_t(r) * a.ls + sg] = ss;
        }
        const unsigned anybad = __ballot_sync(FULL, bad);
        if (lane == 0) {
            uint32_t kx = 0;
#pragma unroll
            for (int j = 0; j < TB; ++j) kx = max(kx, km[j]);
            a.stat[size_t(r) * a.nu + q] = make_uint4(__float_as_uint(um), 0u, anybad ? 1u : 0u, kx);
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) A[j] = Bv[j];
        u = un;
    }
}

// FIN: the summary of input row r into this CTA's tables, as pass 1 and pass1_totals
// leave them in a one-CTA cluster: segment keys (and, with `masses`, segment masses)
// and part[0] = (M; V as the bound of the positive count, bad flag, largest key), and
// with `uhist` the histogram of the units' largest keys (key >> 21) added into uhist,
// which the caller cleared (a block barrier orders the clear before the counts), and
// with `umass` / `ukey` each unit's mass and largest key, with `shist` the histogram of
// the segments' keys (key >> 21) added into shist, cleared by the caller as uhist.  M
// is the sum of the unit masses in a fixed order (thread t adds units t, t + NT, ...
// in turn, then a tree over the lanes and the warps in order).  Every thread issues
// all of its loads before it uses any (one round trip to L2).  The summary was
// written by the previous launch, so it is read through L2 (ld.global.cg).
// Block-collective; ends with a block barrier.
__device__ __forceinline__ void load_summary(const SampleArgs& a, int r, Smem sm, bool masses, int warp, int lane,
                                             int tid, uint32_t* uhist = nullptr, float* umass = nullptr,
                                             uint32_t* ukey = nullptr, uint32_t* shist = nullptr) {
    const uint4* key4 = reinterpret_cast<const uint4*>(a.skey + size_t(r) * a.ls);
    const uint4* mass4 = reinterpret_cast<const uint4*>(a.smass + size_t(r) * a.ls);
    const uint4* st = a.sstat + size_t(r) * a.nu;
    const int n4 = a.ls >> 2;
    float ms = 0.f;
    bool bd = false;
    uint32_t km = 0;
#pragma unroll 1
    for (int i0 = 0; i0 < max(n4, a.nu); i0 += 2 * NT) {
        uint4 k[2], m[2], v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = i0 + h * NT + tid;
            k[h] = i < n4 ? __ldcg(key4 + i) : make_uint4(0u, 0u, 0u, 0u);
            m[h] = (masses && i < n4) ? __ldcg(mass4 + i) : make_uint4(0u, 0u, 0u, 0u);
            v[h] = i < a.nu ? __ldcg(st + i) : make_uint4(0u, 0u, 0u, 0u);
        }
        if ((uhist || shist) && i0 == 0) __syncthreads();  // the caller's clear of the histogram, before any count
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = i0 + h * NT + tid;
            if (i < n4) {
                const uint32_t kk[4] = {k[h].x, k[h].y, k[h].z, k[h].w};
                const uint32_t mm[4] = {m[h].x, m[h].y, m[h].z, m[h].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (4 * i + c < a.ns) {
                        sm.segkey()[4 * i + c] = kk[c];
                        if (masses) sm.mass(0)[4 * i + c] = __uint_as_float(mm[c]);
                        if (shist) atomicAdd(&shist[min(uint32_t(HBINS - 1), kk[c] >> 21)], 1u);
                    }
                }
            }
            ms += __uint_as_float(v[h].x);
            bd |= v[h].z != 0u;
            km = max(km, v[h].w);
            if (uhist && i < a.nu) atomicAdd(&uhist[min(uint32_t(HBINS - 1), v[h].w >> 21)], 1u);
            if (umass && i < a.nu) {
                umass[i] = __uint_as_float(v[h].x);
                ukey[i] = v[h].w;
            }
        }
    }
    ms = warp_sum(ms);
    bd = __any_sync(FULL, bd);
    km = warp_max_u(km);
    float* rf = reinterpret_cast<float*>(sm.red());
    if (lane == 0) {
        rf[warp] = ms;
        sm.red()[NW + warp] = bd ? 1 : 0;
        sm.red()[2 * NW + warp] = int(km);
    }
    __syncthreads();
    if (tid == 0) {
        Part& pt = sm.part()[0];
        float m = 0.f;
        int b = 0;
        uint32_t mk = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            m += rf[w];
            b |= sm.red()[NW + w];
            mk = max(mk, uint32_t(sm.red()[2 * NW + w]));
        }
        pt.f[0] = m;
        pt.u[0] = uint32_t(a.V);  // the scan counts no positives: V bounds the tokens above 0
        pt.u[1] = uint32_t(b);
        pt.u[2] = mk;
    }
    __syncthreads();
}

// FIN: the histogram of this CTA's segment keys (key >> 21) into hist(), which the
// caller cleared.  Block-collective; the caller synchronises before it is read.
__device__ __forceinline__ void summary_hist(Smem sm, int ns, int tid) {
#pragma unroll 1
    for (int i = tid; i < ns; i += NT) atomicAdd(&sm.hist()[min(uint32_t(HBINS - 1), sm.segkey()[i] >> 21)], 1u);
}

// The acceptance test f(tau) ([blog] rejection sampling: count / remaining mass above
// the pivot; [explainer] Top-k, Top-p, Min-p), from the count and the mass of the
// tokens strictly above tau.
struct Pred {
    bool single;  // the one-pivot rule: pivot2 = pivot1 (after a rejection, low <- pivot1)
    bool k_on, p_on, m_on;
    int k;
    float pthr;   // top_p * M'   (M' = M, or F_k for top-k-first)
    float t32;    // min-p threshold: float32 rounded up from min_p * max
    // The second pivot ([blog] dual pivot): the fp32 midpoint of pivot1 and high.
    __device__ __forceinline__ float pivot2(float pivot1, float high) const {
        return single ? pivot1 : (pivot1 + high) * 0.5f;
    }
    __device__ __forceinline__ bool operator()(int cnt, float mass, float tau) const {
        if (k_on && !(cnt < k)) return false;
        if (p_on && !(cnt == 0 || mass < pthr)) return false;
        if (m_on && !(tau >= t32)) return false;
        return true;
    }
};

// The other CTAs: follow the leader's commands until EXIT (or until a collection that
// completed the leader's list).
template <bool VEC>
__device__ __forceinline__ void sample_peer(const float* __restrict__ row, Geom g, Smem sm, int rank,
                                        int C, int warp, int lane, int tid) {
    for (;;) {
        cluster_sync();  // the command is published
        const Ctl c = *sm.ctl();
        if (c.cmd == CMD_PIVOT2) {
            pivot_pass<VEC>(row, g, sm, false, rank, c.f[0], c.f[1], c.ia, c.ib, warp, lane, tid);
        } else if (c.cmd == CMD_SEARCH) {
            const uint64_t hi = uint64_t(c.hi_lo) | (uint64_t(c.hi_hi) << 32);
            search_pass<VEC, true, false>(row, g, sm, false, rank, c.u[0], hi, KeyProb(), warp, lane, tid);
        } else if (c.cmd == CMD_COLLECT) {
            const uint64_t hi = uint64_t(c.hi_lo) | (uint64_t(c.hi_hi) << 32);
            // ib = 1: exact offsets (this CTA's base in bcast[2]); else a region of CAP / C
            const int base = c.ib ? sm.bcast()[2] : rank * (CAP / C);
            collect_own<VEC>(row, g, sm, false, rank, C, base, c.ib ? CAP - base : CAP / C, c.u[0], hi, KeyProb(),
                             false, c.ib == 0, warp, lane, tid);
        } else {
            return;  // CMD_EXIT
        }
        cluster_sync();  // the results are in the leader
        if (c.cmd == CMD_COLLECT) {
            if (c.ib) {
                if (c.flag) return;
            } else {
                const uint64_t hi = uint64_t(c.hi_lo) | (uint64_t(c.hi_hi) << 32);
                const int mode = settle_list<VEC>(row, g, sm, false, rank, C, c.u[0], hi, KeyProb(), false, warp,
                                                  lane, tid);
                if (c.flag && mode >= 0) return;
            }
        }
    }
}

// One compact round on the leader's list (warp-collective): draw, reduce, decide.
// Returns 1 if accepted (token in j), 0 to continue, -1 if the list had no token
// above low (cannot happen while S_low > 0).
__device__ __forceinline__ int compact_round(Smem sm, int n_list, const Pred& f, bool any_filter, float u, float& low,
                                             float& high, float& S_low, int lane, int& j) {
    const int e = locate_in_list(sm.lv(), n_list, low, u * S_low, lane);
    if (e < 0) return -1;
    j = sm.li()[e];
    const float pivot1 = sm.lv()[e];
    if (!any_filter) return 1;
    const float pivot2 = f.pivot2(pivot1, high);
    float M1 = 0.f, M2 = 0.f;
    int C1 = 0, C2 = 0;
    for (int i = lane; i < n_list; i += 32) {
        const float x = sm.lv()[i];
        const bool g1 = x > pivot1, g2 = x > pivot2;
        M1 += g1 ? x : 0.f;
        M2 += g2 ? x : 0.f;
        C1 += g1;
        C2 += g2;
    }
    M1 = warp_sum(M1);
    M2 = warp_sum(M2);
    C1 = warp_sum_i(C1);
    C2 = warp_sum_i(C2);
    if (f(C1, M1, pivot1)) return 1;
    if (f(C2, M2, pivot2)) {
        low = pivot1;
        high = pivot2;
        S_low = M1;
    } else {
        low = pivot2;
        S_low = M2;
    }
    return 0;
}


// The rounds on a short candidate list held in warp 0's registers (kept[r] marks the
// filtered set; S_low its mass): the same draw, fused reduction and three cases as
// compact_round, on registers.  Returns the token (-1 after R_MAX rounds or with
// nothing eligible); the number of rounds in `rounds`.
__device__ __forceinline__ int small_rounds(const Small& s, const bool* kept, const Pred& f, float S_low, float high,
                                            unsigned long long seed, unsigned long long offset, uint32_t b, int lane,
                                            int& rounds, const float* u32 = nullptr) {
    float low = 0.f;
    // Lane l holds the uniform of round l: 32 rounds of the stream at the cost of one
    // (or, with u32, as another warp drew them beforehand).
    const float u_lane = u32 ? u32[lane] : sampler_uniform(seed, offset, b, uint32_t(lane));
#pragma unroll 1
    for (int round = 0; round < R_MAX; ++round) {
        const float u = round < 32 ? __shfl_sync(FULL, u_lane, round) : sampler_uniform(seed, offset, b, uint32_t(round));
        const float target = u * S_low;
        // Inverse transform over the list in index order (lane-major): the lane whose
        // running sum passes the target, then the slot inside it.
        float w[SR], lsum = 0.f;
#pragma unroll
        for (int r = 0; r < SR; ++r) {
            w[r] = kept[r] && s.x[r] > low ? s.x[r] : 0.f;
            lsum += w[r];
        }
        const float incl = warp_incl_scan(lsum, lane);
        const unsigned hit = __ballot_sync(FULL, lsum > 0.f && incl > target);
        const unsigned elig = __ballot_sync(FULL, lsum > 0.f);
        if (!elig) break;
        // In the chosen lane: the first eligible slot whose running sum passes the
        // target, else its last eligible slot (also when no lane passed it).
        const int l = hit ? __ffs(hit) - 1 : 31 - __clz(elig);
        int pick = -1, last = 0;
        float run = incl - lsum;
#pragma unroll
        for (int r = 0; r < SR; ++r) {
            if (w[r] > 0.f) {
                run += w[r];
                last = r;
                if (pick < 0 && run > target) pick = r;
            }
        }
        if (pick < 0 || !hit) pick = last;
        pick = __shfl_sync(FULL, pick, l);
        float xv = 0.f;
        int iv = 0;
#pragma unroll
        for (int r = 0; r < SR; ++r) {
            xv = r == pick ? s.x[r] : xv;
            iv = r == pick ? s.i[r] : iv;
        }
        const float pivot1 = __shfl_sync(FULL, xv, l);
        const int j = __shfl_sync(FULL, iv, l);
        const float pivot2 = f.pivot2(pivot1, high);
        float m1 = 0.f, m2 = 0.f;
        int c1 = 0, c2 = 0;
#pragma unroll
        for (int r = 0; r < SR; ++r) {
            const bool a1 = kept[r] && s.x[r] > pivot1, a2 = kept[r] && s.x[r] > pivot2;
            m1 += a1 ? s.x[r] : 0.f;
            m2 += a2 ? s.x[r] : 0.f;
            c1 += a1;
            c2 += a2;
        }
        const float M1 = warp_sum(m1), M2 = warp_sum(m2);
        const int C1 = warp_sum_i(c1), C2 = warp_sum_i(c2);
        if (f(C1, M1, pivot1)) {
            rounds = round + 1;
            return j;
        }
        if (f(C2, M2, pivot2)) {
            low = pivot1;
            high = pivot2;
            S_low = M1;
        } else {
            low = pivot2;
            S_low = M2;
        }
    }
    rounds = R_MAX;
    return -1;
}



// FIN: the finishing launch after scan_kernel, one CTA per output row (launched as
// one-CTA clusters): the row's summary replaces pass 1, and everything after it runs
// as in a cluster of one.
template <bool VEC, bool SOFT, bool FIN>
__device__ __forceinline__ void sample_row(const SampleArgs& a) {
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool leader = rank == 0;
    const Smem sm(a.ns);
    Geom g(a.V, a.shift, a.ns, a.nsc, rank);
    const int V = a.V, ns = a.ns;
    const KeyProb keyf;

    grid_dependency_wait();
    allow_dependents();
    if (FIN && b == 0 && tid < SCAN_CTRS && a.sctr) a.sctr[tid * SCAN_CTR_STRIDE] = 0u;  // the scan is complete
    // ---- a1: row map and parameters (every CTA reads them)
    const int r = a.indices ? a.indices[b] : b;
    const bool row_ok = r >= 0 && r < a.batch_in;
    const float* row = a.probs + size_t(row_ok ? r : 0) * size_t(V);
    // The logits path picks its pass-1 variant by the row's k and needs 1/T in pass 1;
    // the other parameters are read after pass 1 (below).
    const int k_soft = SOFT && a.top_k ? a.top_k[b] : 0;
    const float temp = SOFT && a.temperature ? a.temperature[b] : 1.f;
    const bool kfirst_soft = SOFT && a.order == 0 && k_soft > 0 && k_soft < V;
    // Pass 1 counts segment maxima into the histogram in every top-k-first launch of
    // probabilities, whatever the row's k, so that the row streams without waiting for
    // its parameters; rows that need no top-k bound leave the counts unused.
    const int hist_sh = (SOFT ? (kfirst_soft && ns >= k_soft) : (a.order == 0 && a.top_k != nullptr)) ? 21 : -1;

    // Rows of logits are read once too: pass 1 keeps, per segment, its largest logit and
    // its mass relative to it (an online softmax); the row's maximum follows from the
    // CTAs' after the barrier.
    if (SOFT) g.vinv = 1.f / temp;

    // ---- a2: pass 1, the only HBM read of the row, inside a split cluster barrier.
    // Its set-up runs once the first loads are in flight: the histograms cleared, the
    // trip counter, the cluster's first arrive; then one lane copies the row's
    // parameters into shared memory, read after the block barrier that follows pass 1.
    auto setup = [&]() {
        if (hist_sh >= 0)
            for (int i = tid; i < HBINS; i += NT) {
                sm.hist()[i] = 0u;
                sm.hist()[HBINS + i] = 0u;
                reinterpret_cast<uint32_t*>(sm.lv())[i] = 0u;
            }
        if (tid == 0) *sm.ctr() = NW;
        __syncthreads();
        cluster_arrive();
        if (tid == NT - 32) {
            uint32_t* pr = sm.prm();
            pr[0] = uint32_t(a.top_k ? a.top_k[b] : 0);
            pr[1] = __float_as_uint(a.top_p ? a.top_p[b] : 1.f);
            pr[2] = __float_as_uint(a.min_p ? a.min_p[b] : 0.f);
            // The row's generator state ([explainer] RNG ownership).
            *reinterpret_cast<unsigned long long*>(pr + 4) = a.seeds ? a.seeds[b] : a.seed;
            *reinterpret_cast<unsigned long long*>(pr + 6) =
                (a.offsets ? a.offsets[b] : a.offset) + (a.offset_dev ? *a.offset_dev : 0ull);
        }
    };
    int pos = 0;
    bool bad = false;
    uint32_t kmax = 0;
    if (FIN) {
        // The same set-up without the cluster arrive: both histograms cleared for a
        // top-k-first launch, the trip counter, the row's parameters.
        if (a.order == 0 && a.top_k)
            for (int i = tid; i < 2 * HBINS; i += NT) sm.hist()[i] = 0u;
        if (tid == 0) *sm.ctr() = NW;
        if (tid == NT - 32) {
            uint32_t* pr = sm.prm();
            pr[0] = uint32_t(a.top_k ? a.top_k[b] : 0);
            pr[1] = __float_as_uint(a.top_p ? a.top_p[b] : 1.f);
            pr[2] = __float_as_uint(a.min_p ? a.min_p[b] : 0.f);
            *reinterpret_cast<unsigned long long*>(pr + 4) = a.seeds ? a.seeds[b] : a.seed;
            *reinterpret_cast<unsigned long long*>(pr + 6) =
                (a.offsets ? a.offsets[b] : a.offset) + (a.offset_dev ? *a.offset_dev : 0ull);
        }
        // The summary's loads go out with the parameters' (logit rows without a top-k
        // bound replace the tables with a pass over the row below).
        if (row_ok) load_summary(a, r, sm, !SOFT && a.smass != nullptr, warp, lane, tid);
    } else if (row_ok) {
        if (SOFT && kfirst_soft)  // draws come from the gathered candidates: keys only
            pass1<VEC, true, false, 1>(row, g, sm, hist_sh, warp, lane, pos, bad, kmax, setup);
        else if (SOFT)
            pass1<VEC, true, false, 2>(row, g, sm, -1, warp, lane, pos, bad, kmax, setup);
        else
            pass1<VEC, true, true>(row, g, sm, hist_sh, warp, lane, pos, bad, kmax, setup);
    } else {
        setup();
        for (int i = g.s0 + tid; i < g.s1; i += NT) {
            sm.segkey()[i] = 0u;
            sm.mass(0)[i] = 0.f;
        }
    }
    __syncthreads();  // the row's parameters
    const int k = int(sm.prm()[0]);
    const float tp = __uint_as_float(sm.prm()[1]);
    const float mp = __uint_as_float(sm.prm()[2]);
    const unsigned long long seed_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 4);
    const unsigned long long offset_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 6);
    const uint32_t stream_b = a.seeds ? 0u : uint32_t(b);
    const bool k_on = k > 0 && k < V;
    const bool kfirst = a.order == 0 && k_on;
    const bool need_hist = kfirst && ns >= k;
    if (FIN) {
        if (!row_ok) {
            for (int i = tid; i < ns; i += NT) {
                sm.segkey()[i] = 0u;
                sm.mass(0)[i] = 0.f;
            }
            if (tid == 0) sm.part()[0] = Part{};
        } else if (!kfirst && (SOFT || !a.smass)) {
            // A draw over the whole row needs segment masses, which this summary does not
            // hold (masses of logits also depend on the row's temperature): this row (no
            // top-k bound in a top-k-first launch) is read again here, from L2, as pass 1
            // reads it.
            if (SOFT) {
                pass1<VEC, true, false, 2>(row, g, sm, -1, warp, lane, pos, bad, kmax);
            } else {
                pass1<VEC, true, true>(row, g, sm, -1, warp, lane, pos, bad, kmax);
            }
            pass1_totals(g, sm, true, 0, 1, pos, bad, kmax, -1, true, true, warp, lane, tid, SOFT, 0);
        } else if (need_hist) {
            summary_hist(sm, ns, tid);  // the tables were loaded with the parameters
        }
        __syncthreads();  // the tables, part[0] and the histogram
    } else {
        cluster_wait();  // every CTA has started and cleared its histogram
        pass1_totals(g, sm, leader, rank, C, pos, bad, kmax, need_hist ? 21 : -1, !(SOFT && kfirst), !kfirst, warp,
                     lane, tid, SOFT && !kfirst, need_hist ? k : 0);
        cluster_sync();  // the leader's segment table, every CTA's parts and histogram, are complete
    }

    // Rows of logits: the row's largest logit m (the CTAs' maxima are logit keys in
    // part[].u[2]) and each CTA's factor exp((m_c - m) / T) from its maximum to the row's,
    // in scale[c].  From here on the row is read as the weights w = exp((z - m) / T).
    float* scale = reinterpret_cast<float*>(sm.red() + 112);  // [MAX_CLUSTER], past the search scratch
    uint32_t row_mkey = 0;
    if (SOFT) {
        row_mkey = warp_max_u(lane < C ? sm.part()[lane].u[2] : 0u);
        const bool fin = row_mkey > 0x007fffffu && row_mkey < 0xff800000u;
        g.vm = from_logit_key(row_mkey);
        g.soft = true;
        if (tid < C) {
            const uint32_t kc = sm.part()[tid].u[2];
            scale[tid] = (fin && kc > 0x007fffffu) ? expf((from_logit_key(kc) - g.vm) * g.vinv) : 0.f;
        }
        if (!kfirst) soft_segment_keys(g, sm, tid);
        __syncthreads();
    }

    // ---- a3 (first half, every CTA): top-k-first candidates.  Every CTA derives the
    // same lower bound L0 <= t_k from its copy of the histogram and sends its elements
    // >= L0 to its region of the leader's list.
    int list_mode = -1;  // 0: regions fit, 1: contiguous, -1: no list (too many / not top-k-first)
    uint32_t L0 = 1u;
    Totals tot;
    if (kfirst) {
        const uint32_t mk = warp_max_u(lane < C ? sm.part()[lane].u[2] : 0u);
        L0 = max(1u, need_hist ? hist_bound(sm, g, rank, C, k, mk, warp, lane, tid) : 0u);
        if (SOFT) {  // the segment keys and the bound, from logits to weights
            soft_segment_keys(g, sm, tid);
            L0 = soft_bound(g, L0);
            __syncthreads();
        }
        collect_own<VEC>(row, g, sm, leader, rank, C, rank * (CAP / C), CAP / C, L0, NO_LIMIT, keyf, false, true,
                         warp, lane, tid);
        if (leader) {  // the row's totals while the other CTAs finish their candidates
            cluster_arrive();
            tot = cluster_totals(sm, C);
            cluster_wait();
        } else {
            cluster_sync();
        }
        // every region and count is in
        list_mode = settle_list<VEC>(row, g, sm, leader, rank, C, L0, NO_LIMIT, keyf, false, warp, lane, tid);
    } else if (leader) {
        tot = cluster_totals(sm, C);
    }
    if (!leader) {
        if (list_mode < 0) sample_peer<VEC>(row, g, sm, rank, C, warp, lane, tid);
        return;
    }

    // ---- leader from here on
    Pred f;
    f.single = a.single_pivot != 0;
    f.k_on = k_on;
    f.k = k;
    f.p_on = tp < 1.f;
    f.m_on = mp > 0.f;
    f.pthr = 0.f;
    f.t32 = 0.f;
    const bool any_filter = f.k_on || f.p_on || f.m_on;

    if (SOFT) {  // the CTAs' masses to the row's maximum; the largest weight is exp(0) = 1
        const bool inC = lane < C;
        const bool fin = row_mkey > 0x007fffffu && row_mkey < 0xff800000u;
        // top-k-first kept no masses: the row's mass only decides validity there, and is
        // at least the largest weight, 1
        tot.M = kfirst ? (fin ? 1.f : 0.f) : warp_sum(inC ? scale[lane] * sm.part()[lane].f[0] : 0.f);
        tot.maxkey = fin ? 0x3f800000u : 0u;
        if (!kfirst)  // the segment table for draws over the whole row, from each CTA's maximum to the row's
            for (int i = tid; i < ns; i += NT) sm.mass(0)[i] *= scale[i / a.nsc];
    }
    const int npos = tot.npos;
    const bool any_bad = tot.any_bad;
    const float M = tot.M;   // sum of the per-CTA ordered sums
    const uint32_t maxkey = tot.maxkey;
    if (tid < C) sm.cmass()[tid] = SOFT ? scale[tid] * sm.part()[tid].f[0] : sm.part()[tid].f[0];
    const float rowmax = __uint_as_float(maxkey);
    bool valid = row_ok && !isnan(tp) && !isnan(mp) && !any_bad && M > 0.f && M <= 3.402823466e38f &&
                 (!SOFT || temp > 0.f);
    if (f.m_on) {
        f.t32 = __double2float_ru(double(mp) * double(rowmax));
        if (!(rowmax >= f.t32)) valid = false;  // S is empty: f(max) = 0
    }
    if (list_mode < 0) __syncthreads();

    bool peers = list_mode < 0;  // the other CTAs still wait for commands
    auto dismiss = [&]() {
        if (peers) {
            Ctl c{};
            c.cmd = CMD_EXIT;
            send_command(sm, c, C, tid);
            peers = false;
        }
    };

    int token = -1, rounds = 0;
    bool accepted = false;
    if (valid) {
        float low = 0.f, high = rowmax, S_low = M;
        int cur = 0;            // mass(cur)[s] = mass of segment s above `low`
        int count_low = npos;   // tokens above `low`
        int low_u = -1;         // part[c].u[low_u]: CTA c's exact count above `low` (-1: not known)
        int n_list = 0;
        bool compact = false;
        f.pthr = tp * M;

        // ---- a3 (second half, leader): t_k and F_k
        if (kfirst && list_mode >= 0 && regions_total(sm, C) <= SMALL) {
            // The usual case: a short candidate list, finished in warp 0's registers.
            if (warp == 0) {
                const Small sl = small_gather(sm, C, CAP / C, list_mode == 1, lane);
                const uint32_t tk = small_kth(sl, k, keyf);
                bool kept[SR];
                float fk = 0.f;
#pragma unroll
                for (int r = 0; r < SR; ++r) {
                    kept[r] = sl.in[r] && keyf(sl.x[r]) >= tk;
                    fk += kept[r] ? sl.x[r] : 0.f;
                }
                const float Fk = warp_sum(fk);
                f.pthr = tp * Fk;  // top-p inside the k, measured against F_k
                token = small_rounds(sl, kept, f, Fk, high, seed_b, offset_b, stream_b, lane, rounds);
                accepted = token >= 0;
            }
        } else {
        if (kfirst) {
            int n = -1;
            if (list_mode >= 0) {
                n = regions_total(sm, C);
                if (list_mode == 0 && warp == 0) join_regions_warp(sm, C, CAP / C, lane);
            }
            if (n >= 0) {
                compact = true;
                // The list holds every element >= L0, hence every element >= t_k.
                __syncthreads();  // the joined list
                const uint32_t tk = kth_key_cta(sm, n, k, keyf, warp, lane, tid);
                if (warp == 0) {
                    n_list = filter_list_warp(sm, n, tk, keyf, lane);
                    float s = 0.f;
                    for (int i = lane; i < n_list; i += 32) s += sm.lv()[i];
                    S_low = warp_sum(s);
                }
                low = 0.f;
            } else {
                // Too many candidates: t_k by a threshold search with the cluster.
                Search st = search_start(maxkey, M, V);
                threshold_search<VEC, true, false, false>(row, g, sm, C, st, k, 0.f, keyf, warp, lane, tid);
                const uint32_t tk = uint32_t(st.lo);
                low = tk >= 1u ? __uint_as_float(tk - 1u) : 0.f;  // x > low  <=>  key(x) >= t_k
                // Per-segment and per-CTA masses above `low` for the draws (both pivots = low).
                Ctl c{};
                c.cmd = CMD_PIVOT2;
                c.f[0] = low;
                c.f[1] = low;
                c.ia = 0;
                c.ib = 1;
                send_command(sm, c, C, tid);
                pivot_pass<VEC>(row, g, sm, true, 0, low, low, 0, 1, warp, lane, tid);
                cluster_sync();
                {
                    const bool inC = lane < C;
                    const Part& pc = sm.part()[inC ? lane : 0];
                    count_low = warp_sum_i(inC ? int(pc.u[0]) : 0);
                    low_u = 0;
                    S_low = warp_sum(inC ? pc.f[0] : 0.f);
                }
                if (tid < C) sm.cmass()[tid] = sm.part()[tid].f[0];
                __syncthreads();
                cur = 0;
            }
            f.pthr = tp * S_low;  // top-p inside the k, measured against F_k
        }

        // ---- a4..a7: rejection rounds
        for (int round = 0; round < R_MAX; ++round) {
            if (!compact && count_low <= CAP) {
                // Few tokens left above `low`: gather them; the leader goes on alone.
                n_list = gather_leader<VEC>(row, g, sm, C, prob_key(low) + 1u, NO_LIMIT, keyf, true, warp, lane, tid,
                                            low_u);
                if (n_list >= 0) peers = false;  // they left with the completed list
                dismiss();
                if (n_list < 0) break;
                compact = true;
            }
            const float u = sampler_uniform(seed_b, offset_b, stream_b, uint32_t(round));
            if (compact) {
                if (warp != 0) break;
                int j = -1;
                const int st = compact_round(sm, n_list, f, any_filter, u, low, high, S_low, lane, j);
                if (st < 0) break;
                if (st > 0) {
                    accepted = true;
                    token = j;
                    rounds = round + 1;
                    break;
                }
                continue;
            }
            // ---- a5: draw (warp 0): owner CTA, segment, token
            if (warp == 0) {
                const unsigned long long jx = draw_full<VEC>(row, g, sm, C, cur, low, u * S_low, lane);
                if (lane == 0) {
                    sm.red()[32] = unpack_j(jx);
                    reinterpret_cast<float*>(sm.red())[33] = unpack_x(jx);
                }
            }
            __syncthreads();
            const int j = sm.red()[32];
            const float pivot1 = reinterpret_cast<float*>(sm.red())[33];
            __syncthreads();
            if (j < 0) break;
            if (!any_filter) {
                accepted = true;
                token = j;
                rounds = round + 1;
                break;
            }
            const float pivot2 = f.pivot2(pivot1, high);

            // ---- a6: fused (mass, count) above pivot1 and pivot2, on the whole cluster
            const int ia = cur == 0 ? 1 : 0;
            const int ib = cur == 2 ? 1 : 2;
            Ctl c{};
            c.cmd = CMD_PIVOT2;
            c.f[0] = pivot1;
            c.f[1] = pivot2;
            c.ia = ia;
            c.ib = ib;
            send_command(sm, c, C, tid);
            pivot_pass<VEC>(row, g, sm, true, 0, pivot1, pivot2, ia, ib, warp, lane, tid);
            cluster_sync();  // every part is in
            const bool inC = lane < C;
            const Part& pc = sm.part()[inC ? lane : 0];
            const int C1 = warp_sum_i(inC ? int(pc.u[0]) : 0);
            const int C2 = warp_sum_i(inC ? int(pc.u[1]) : 0);
            const float M1 = warp_sum(inC ? pc.f[0] : 0.f);
            const float M2 = warp_sum(inC ? pc.f[1] : 0.f);

            // ---- a7: the three cases
            if (f(C1, M1, pivot1)) {
                accepted = true;
                token = j;
                rounds = round + 1;
                break;
            }
            const bool narrow = f(C2, M2, pivot2);
            if (narrow) {
                low = pivot1;
                high = pivot2;
                S_low = M1;
                count_low = C1;
                low_u = 0;
                cur = ia;
            } else {
                low = pivot2;
                S_low = M2;
                count_low = C2;
                low_u = 1;
                cur = ib;
            }
            if (tid < C) sm.cmass()[tid] = narrow ? sm.part()[tid].f[0] : sm.part()[tid].f[1];
            __syncthreads();
        }
        if (!accepted) rounds = R_MAX;
        }
    }

    // ---- a8: outputs (the peers are let go first; warp 0 holds the result)
    if (peers) dismiss();
    if (tid == 0) {
        a.out_token[b] = accepted ? token : -1;
        a.out_valid[b] = accepted ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = rounds;
    }
}

template <bool VEC, bool SOFT, bool FIN>
__global__ void __launch_bounds__(NT, FIN ? 2 : 3) sample_kernel(const SampleArgs a) {
    sample_row<VEC, SOFT, FIN>(a);
}

// The whole finishing path of one row, out of line: the lean top-k-first kernel's
// fallback for rows outside its fast case.
template <bool VEC>
FS_COLD __device__ void sample_row_fin(const SampleArgs& a) {
    sample_row<VEC, false, true>(a);
}

// ------------------------------------------------------------------ lean top-k-first finish

// The finishing launch of the top-k-first samplers on rows of probabilities, for the
// usual row.  The bound uk: the lower edge of the histogram bin (key >> 21, a quarter
// binade) that holds the k-th largest of the units' maxima.  The units' maxima are a
// subset of the row, and the k-th largest of a subset is at most the row's own
// ([explainer] filter order: t_k is the k-th largest value), so uk <= t_k: every
// element >= t_k lies in a segment whose maximum is >= uk.  Steps, with two round
// trips to L2 after the scan: (1) the row's summary, the histogram of its unit maxima
// counted as it is unpacked, uk; (2) the live segments (maximum >= uk) copied in index
// order into shared memory, their elements >= uk written in index order into the
// candidate list; then warp 0 finds t_k and runs the rejection rounds in registers as
// the cluster's leader does.  The work is spread so that no warp runs a long chain of
// dependent instructions: this code runs once per launch at one CTA per SM, where such
// chains, not memory, set the time.  Any other row (a bad row index, no top-k filter,
// fewer units than k, segments of several blocks, more than KF_LIVE live segments or
// more than SMALL candidates) takes the general finishing path, out of line.
constexpr int KF_LIVE = 112;  // live segments the lean finish stages (fpt = 15 float4 per thread at most)

// The staging area of the lean finish (KF_LIVE blocks), after the carve-up.
__host__ __device__ inline size_t kfirst_smem(int ns) { return Layout(ns).total() + size_t(KF_LIVE) * BLK * 4; }
__device__ __forceinline__ float* kfirst_stage(Smem sm) {
    return reinterpret_cast<float*>(smem_raw + Layout(sm.ns).total());
}

template <bool VEC>
__global__ void __launch_bounds__(NT, 2) kfirst_kernel(const SampleArgs a) {
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Smem sm(a.ns);
    const int V = a.V, ns = a.ns, nu = a.nu;
    const KeyProb keyf;
    // The row index and the parameters are read before the dependency wait: they were
    // written before the scan of this call started (the scan waits for its own
    // predecessors before it lets this launch begin), and only the summary comes from
    // the scan.
    const int r = a.indices ? a.indices[b] : b;
    const bool row_ok = r >= 0 && r < a.batch_in;
    if (tid == NT - 32) {
        uint32_t* pr = sm.prm();
        pr[0] = uint32_t(a.top_k ? a.top_k[b] : 0);
        pr[1] = __float_as_uint(a.top_p ? a.top_p[b] : 1.f);
        pr[2] = __float_as_uint(a.min_p ? a.min_p[b] : 0.f);
        *reinterpret_cast<unsigned long long*>(pr + 4) = a.seeds ? a.seeds[b] : a.seed;
    }
    for (int i = tid; i < HBINS; i += NT) sm.hist()[i] = 0u;
    grid_dependency_wait();
    allow_dependents();
    if (b == 0 && tid < SCAN_CTRS && a.sctr) a.sctr[tid * SCAN_CTR_STRIDE] = 0u;  // the scan is complete
    if (tid == NT - 32) {  // a device-resident offset may be advanced by the kernel before
        *reinterpret_cast<unsigned long long*>(sm.prm() + 6) =
            (a.offsets ? a.offsets[b] : a.offset) + (a.offset_dev ? *a.offset_dev : 0ull);
    }
    // ---- (1) the summary, with the histogram of the unit maxima; the bound
    if (row_ok) {
        load_summary(a, r, sm, false, warp, lane, tid, sm.hist());  // ends with a block barrier
    } else {
        __syncthreads();
    }
    const int k = int(sm.prm()[0]);
    if (!row_ok || !(k > 0 && k < V) || nu < k || a.shift != 0) {
        __syncthreads();
        sample_row_fin<VEC>(a);
        return;
    }
    if (warp == 0) {
        // The bin holding the k-th largest unit maximum, from the top: its lower edge is
        // at most that maximum, hence at most t_k.
        uint32_t above;
        const int B = scan_bins_down<uint32_t>(sm.hist(), int(min(uint32_t(HBINS - 1), sm.part()[0].u[2] >> 21)),
                                               uint32_t(k), lane, above);
        if (lane == 0) sm.bcast()[0] = max(B, 0);
    }
    __syncthreads();
    const uint32_t uk = max(1u, uint32_t(sm.bcast()[0]) << 21);  // zeros are never candidates
    // ---- (2) the live segments (maximum >= uk), copied into the staging area in index
    // order, then the candidates.  Each warp first counts the live segments of its
    // contiguous share, so that it knows where its copies start.
    int r0, r1;
    warp_range(ns, warp, r0, r1);
    int nl = 0;
#pragma unroll 1
    for (int b0 = r0; b0 < r1; b0 += 32)
        nl += __popc(__ballot_sync(FULL, b0 + lane < r1 && sm.segkey()[b0 + lane] >= uk));
    if (lane == 0) sm.red()[warp] = nl;
    __syncthreads();
    int off = 0, L = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const int c = sm.red()[w];
        off += w < warp ? c : 0;
        L += c;
    }
    if (L > KF_LIVE) {
        __syncthreads();
        sample_row_fin<VEC>(a);
        return;
    }
    const float* row = a.probs + size_t(r) * size_t(V);
    float* stg = kfirst_stage(sm);
    int* seg = reinterpret_cast<int*>(sm.list());  // [L] the staged segments, in index order
#pragma unroll 1
    for (int b0 = r0; b0 < r1; b0 += 32) {
        unsigned bal = __ballot_sync(FULL, b0 + lane < r1 && sm.segkey()[b0 + lane] >= uk);
#pragma unroll 1
        while (bal) {
            const int sg = b0 + __ffs(bal) - 1;
            bal &= bal - 1u;
            stage4<VEC>(stg + off * BLK + lane * 4, row, V, sg * BLK + lane * 4);
            if (lane == 0) seg[off] = sg;
            ++off;
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();  // every warp's copies and segment numbers
    // Candidates: thread t takes fpt consecutive staged float4 (fpt odd: the eight lanes
    // of a 16-byte access phase then touch eight different bank groups), one block-wide
    // scan of the counts gives every kept value its place in index order.  Rolled loops
    // and few instructions: this code runs once per launch.  Zeros (and the zeros past
    // V) are below uk >= 1; for values >= 0, key >= uk is x >= the float of uk.
    const float ukf = __uint_as_float(uk);
    const int g4 = L * 32;  // staged float4
    const int fpt = ((g4 + NT - 1) / NT) | 1;
    const int g0 = min(g4, tid * fpt), g1 = min(g4, g0 + fpt);
    const float4* stg4 = reinterpret_cast<const float4*>(stg);
    unsigned long long kmask = 0ull;  // 4 bits per float4 of the thread's range (fpt <= 17)
#pragma unroll 1
    for (int g = g0; g < g1; ++g) {
        const float4 x = stg4[g];
        const unsigned m = (x.x >= ukf ? 1u : 0u) | (x.y >= ukf ? 2u : 0u) | (x.z >= ukf ? 4u : 0u) |
                           (x.w >= ukf ? 8u : 0u);
        kmask |= (unsigned long long)m << (4 * (g - g0));
    }
    // Meanwhile the last warp draws the uniforms of the first 32 rounds.
    float* uni = reinterpret_cast<float*>(sm.red()) + (REDW - 32);  // [32]
    if (warp == NW - 1) {
        const unsigned long long seed_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 4);
        const unsigned long long offset_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 6);
        uni[lane] = sampler_uniform(seed_b, offset_b, a.seeds ? 0u : uint32_t(b), uint32_t(lane));
    }
    const int kc = __popcll(kmask);
    const int kincl = warp_incl_scan_i(kc, lane);
    if (lane == 31) sm.red()[warp] = kincl;
    __syncthreads();
    const int wtot = lane < NW ? sm.red()[lane] : 0;
    const int wincl = warp_incl_scan_i(wtot, lane);
    const int n = __shfl_sync(FULL, wincl, NW - 1);
    if (n > SMALL) {
        __syncthreads();
        sample_row_fin<VEC>(a);
        return;
    }
    int pos = __shfl_sync(FULL, wincl - wtot, warp) + kincl - kc;
#pragma unroll 1
    while (kmask) {
        const int bit = __ffsll(kmask) - 1;
        kmask &= kmask - 1ull;
        const int g = g0 + (bit >> 2), q = bit & 3;
        sm.lv()[pos] = stg[4 * g + q];
        sm.li()[pos] = seg[g >> 5] * BLK + (g & 31) * 4 + q;
        ++pos;
    }
    __syncthreads();
    // t_k: every candidate counts the candidates at or above it (the warps holding
    // candidates; broadcast reads, four independent sums); the largest with at least k
    // is t_k (0 when there are fewer than k: the row has fewer than k positives).
    {
        uint32_t best = 0u;
        if (warp * 32 < n) {
            const uint4* c4 = reinterpret_cast<const uint4*>(sm.lv());
            const uint32_t mine = tid < n ? __float_as_uint(sm.lv()[tid]) : 0xffffffffu;
            int gc[4] = {0, 0, 0, 0};
#pragma unroll 1
            for (int t = 0; 4 * t < n; t += 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 w = c4[t + c];  // SMALL entries are always in the list's storage
                    const int e = 4 * (t + c);
                    gc[c] += (w.x >= mine && e < n) + (w.y >= mine && e + 1 < n) + (w.z >= mine && e + 2 < n) +
                             (w.w >= mine && e + 3 < n);
                }
            }
            const int ge = (gc[0] + gc[1]) + (gc[2] + gc[3]);
            best = (tid < n && ge >= k) ? mine : 0u;
            best = warp_max_u(best);
        }
        if (lane == 0) sm.red()[3 * NW + warp] = int(best);
        __syncthreads();
    }
    if (warp != 0) return;
    // ---- warp 0: F_k, the rounds, the outputs (as the cluster's leader)
    const float tp = __uint_as_float(sm.prm()[1]);
    const float mp = __uint_as_float(sm.prm()[2]);
    const unsigned long long seed_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 4);
    const unsigned long long offset_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 6);
    const uint32_t stream_b = a.seeds ? 0u : uint32_t(b);
    const float M = sm.part()[0].f[0];
    const bool any_bad = sm.part()[0].u[1] != 0u;
    const float rowmax = __uint_as_float(sm.part()[0].u[2]);
    Pred f;
    f.single = a.single_pivot != 0;
    f.k_on = true;
    f.k = k;
    f.p_on = tp < 1.f;
    f.m_on = mp > 0.f;
    f.pthr = 0.f;
    f.t32 = 0.f;
    bool valid = !isnan(tp) && !isnan(mp) && !any_bad && M > 0.f && M <= 3.402823466e38f;
    if (f.m_on) {
        f.t32 = __double2float_ru(double(mp) * double(rowmax));
        if (!(rowmax >= f.t32)) valid = false;
    }
    int token = -1, rounds = 0;
    if (valid) {
        Small sl;
        sl.n = n;
#pragma unroll
        for (int q = 0; q < SR; ++q) {
            const int e = SR * lane + q;
            sl.in[q] = e < n;
            sl.x[q] = sl.in[q] ? sm.lv()[e] : 0.f;
            sl.i[q] = sl.in[q] ? sm.li()[e] : 0;
        }
        uint32_t tk = 0u;
#pragma unroll
        for (int w = 0; w < NW; ++w) tk = max(tk, uint32_t(sm.red()[3 * NW + w]));
        bool kp[SR];
        float fk = 0.f;
#pragma unroll
        for (int q = 0; q < SR; ++q) {
            kp[q] = sl.in[q] && keyf(sl.x[q]) >= tk;
            fk += kp[q] ? sl.x[q] : 0.f;
        }
        const float Fk = warp_sum(fk);
        f.pthr = tp * Fk;  // top-p inside the k, measured against F_k
        token = small_rounds(sl, kp, f, Fk, rowmax, seed_b, offset_b, stream_b, lane, rounds, uni);
    }
    if (lane == 0) {
        a.out_token[b] = token >= 0 ? token : -1;
        a.out_valid[b] = token >= 0 ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = rounds;
    }
}

// ------------------------------------------------------------------ lean joint finish
//
// The finishing launch of the joint order with a top-k or a min-p filter on rows of
// probabilities, one CTA per output row.  Each round ([blog] dual-pivot rejection
// sampling) needs a draw over {p > low} in index order and the count and mass above
// both pivots.  Both come from a list in shared memory whenever the list holds every
// element above `low` (above the pivot, for f):
//  * jmode 1 (rows that fit the shared memory): the whole row, staged once;
//  * jmode 0: first the candidates, the elements at or above uk, the larger of the
//    lower edge of the histogram bin (key >> 21) that holds the k-th largest block
//    maximum (so that uk <= t_k: the block maxima are a subset of the row;
//    [explainer] filter order) and the min-p threshold.  Below uk f fails without a
//    count: at least k elements lie above any threshold there, or min-p fails.  A draw
//    while low < uk needs each unit's mass above low: the scan's unit masses while
//    low = 0 (that draw is made by warp 0 during the set-up), else one pass over the
//    row through L2, which also copies every float4 run that holds an element above
//    low into the second list; from then on every round runs on that list, since low
//    never decreases.  If the second list overflows, the next draw below its
//    threshold passes over the row again.
// A list is a sequence of float4 runs of the row in index order (with the index of
// each run's first element, or implied), cut into chunks of 32 runs; the pass that
// evaluates f gives every chunk's mass above both pivots, which is the table of the
// next round's draw.  Other rows (a bad row index, segments of several blocks, in
// jmode 0 neither a top-k bound (a valid k, at most as many as the blocks) nor
// min-p, or a candidate list that overflows or, bounded by the top-k bound alone,
// counts fewer than k elements) take the general finishing path, out of line.

constexpr int JCH = 512;   // chunks of a list, at most
constexpr int JX4 = 1024;  // runs of the candidate list (JX4 / NW per warp)

// The area after the carve-up: the two chunk-mass tables, the chunk bases (run
// offsets) and the chunk maxima, JCH words each; then, in jmode 1, the row; in jmode 0
// the candidate list (JX4 runs and their indices) and the second list (jy4 runs and
// their indices).
__host__ __device__ inline size_t jtab_off(int ns) { return Layout(ns).total(); }
__host__ __device__ inline size_t jx_off(int ns) { return jtab_off(ns) + 4 * size_t(JCH) * 4; }
__host__ __device__ inline size_t jy_off(int ns) { return jx_off(ns) + size_t(JX4) * 20; }

// A list of runs: chunk c is v4[jb[c] .. jb[c] + 32).
struct JList {
    const float4* v4;
    const int* ix;  // element index of each run's .x (nullptr: run i holds elements 4 i .. 4 i + 3)
    int nch;        // chunks
    float lo;       // every element above lo is in the list
};

__device__ __forceinline__ unsigned lanes_below(int lane) { return (1u << lane) - 1u; }

// Appends the lane's run v (elements base .. base + 3) to a warp's slice s4 / si when
// one of its values is above thr, the warp's runs in lane order.  wn counts the warp's
// runs, past the slice's capacity cap too (nothing is written there).  Warp-collective.
__device__ __forceinline__ void append_run(const float4& v, int base, float thr, float4* s4, int* si, int cap, int& wn,
                                           int lane) {
    const bool any = (v.x > thr) | (v.y > thr) | (v.z > thr) | (v.w > thr);
    const unsigned bal = __ballot_sync(FULL, any);
    const int pos = wn + __popc(bal & lanes_below(lane));
    if (any && pos < cap) {
        s4[pos] = v;
        si[pos] = base;
    }
    wn += __popc(bal);
}

// Closes a list kept in slices (warp w's wn_w runs from run w * cap on): each slice
// padded with zero runs to whole chunks, the chunk bases jb in slice order and the
// chunk maxima jk.  Returns the chunk count, or -1 with the tables untouched when a
// slice overflowed or the chunks exceed JCH.  Block-collective.
__device__ __forceinline__ int close_list(float4* v4, int cap, int wn, int* jb, float* jk, Smem sm, int warp,
                                          int lane) {
    int* rw = sm.red() + 56;  // [NW]
    if (lane == 0) rw[warp] = wn;
    __syncthreads();
    int before = 0, total = 0;
    bool over = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const int c = rw[w];
        over |= c > cap;
        const int nc = (min(c, cap) + 31) >> 5;
        before += w < warp ? nc : 0;
        total += nc;
    }
    __syncthreads();  // every thread has read rw
    if (over || total > JCH) return -1;
    const int nc = (wn + 31) >> 5;
    float4* s4 = v4 + size_t(warp) * cap;
    for (int e = wn + lane; e < nc * 32; e += 32) s4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncwarp();
#pragma unroll 1
    for (int i = 0; i < nc; ++i) {
        const float4 v = s4[32 * i + lane];
        const uint32_t m = warp_max_u(prob_key(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w))));
        if (lane == 0) {
            jb[before + i] = warp * cap + 32 * i;
            jk[before + i] = __uint_as_float(m);
        }
    }
    __syncthreads();
    return total;
}

// Every chunk's mass above t1 (m1c) and above t2 (m2c), and the totals: the masses
// summed in a fixed order, the counts exact.  A chunk whose largest value is at most
// min(t1, t2) holds nothing above either and is not read.  When more than DENSE
// threads own a chunk to read, thread c takes chunk c (and c + NT): its 32 runs in an
// order rotated by the lane, so that the eight lanes of an access phase read eight
// different bank groups, and no shuffles; otherwise warp w takes chunks w, w + NW, ...
// four at a time, one run per lane, the four chunks' reductions interleaved.  Each
// thread (warp) adds its chunks in order, then the warps in order.  Block-collective;
// every thread gets the totals.
constexpr int DENSE = 64;
__device__ __forceinline__ void chunk_pass(const JList& L, const int* jb, const float* jk, float t1, float t2,
                                           float* m1c, float* m2c, Smem sm, int tid, int warp, int lane, float& m1,
                                           float& m2, int& c1, int& c2) {
    const float tmin = fminf(t1, t2);
    bool own = false;
    for (int c = tid; c < L.nch; c += NT) own |= jk[c] > tmin;
    const bool dense = __syncthreads_count(own) > DENSE;
    float s1 = 0.f, s2 = 0.f;
    int n1 = 0, n2 = 0;
    if (dense) {
#pragma unroll 1
        for (int c = tid; c < L.nch; c += NT) {
            float a1 = 0.f, a2 = 0.f, b1 = 0.f, b2 = 0.f;
            int k1 = 0, k2 = 0;
            if (jk[c] > tmin) {
                const float4* q = L.v4 + jb[c];
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const float4 v = q[(i + lane) & 31];
                    a1 += (v.x > t1 ? v.x : 0.f) + (v.y > t1 ? v.y : 0.f);
                    b1 += (v.z > t1 ? v.z : 0.f) + (v.w > t1 ? v.w : 0.f);
                    a2 += (v.x > t2 ? v.x : 0.f) + (v.y > t2 ? v.y : 0.f);
                    b2 += (v.z > t2 ? v.z : 0.f) + (v.w > t2 ? v.w : 0.f);
                    k1 += int(v.x > t1) + int(v.y > t1) + int(v.z > t1) + int(v.w > t1);
                    k2 += int(v.x > t2) + int(v.y > t2) + int(v.z > t2) + int(v.w > t2);
                }
            }
            m1c[c] = a1 + b1;
            m2c[c] = a2 + b2;
            s1 += a1 + b1;
            s2 += a2 + b2;
            n1 += k1;
            n2 += k2;
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        n1 = warp_sum_i(n1);
        n2 = warp_sum_i(n2);
    } else {
#pragma unroll 1
        for (int c0 = warp; c0 < L.nch; c0 += 4 * NW) {
            bool act[4];
            bool any = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = c0 + i * NW;
                act[i] = c < L.nch && jk[c] > tmin;
                any |= act[i];
            }
            float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
            int k1[4] = {0, 0, 0, 0}, k2[4] = {0, 0, 0, 0};
            if (any) {  // warp-uniform
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = act[i] ? L.v4[jb[c0 + i * NW] + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                    a1[i] = ((v.x > t1 ? v.x : 0.f) + (v.y > t1 ? v.y : 0.f)) +
                            ((v.z > t1 ? v.z : 0.f) + (v.w > t1 ? v.w : 0.f));
                    a2[i] = ((v.x > t2 ? v.x : 0.f) + (v.y > t2 ? v.y : 0.f)) +
                            ((v.z > t2 ? v.z : 0.f) + (v.w > t2 ? v.w : 0.f));
                    k1[i] = int(v.x > t1) + int(v.y > t1) + int(v.z > t1) + int(v.w > t1);
                    k2[i] = int(v.x > t2) + int(v.y > t2) + int(v.z > t2) + int(v.w > t2);
                }
#pragma unroll
                for (int m = 16; m; m >>= 1) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a1[i] += __shfl_xor_sync(FULL, a1[i], m);
                        a2[i] += __shfl_xor_sync(FULL, a2[i], m);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    k1[i] = __reduce_add_sync(FULL, k1[i]);
                    k2[i] = __reduce_add_sync(FULL, k2[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = c0 + i * NW;
                if (c < L.nch) {
                    if (lane == 0) {
                        m1c[c] = a1[i];
                        m2c[c] = a2[i];
                    }
                    s1 += a1[i];
                    s2 += a2[i];
                    n1 += k1[i];
                    n2 += k2[i];
                }
            }
        }
    }
    float* rf = reinterpret_cast<float*>(sm.red()) + 24;  // [NW] s1, [NW] s2
    int* ri = sm.red() + 24 + 2 * NW;                     // [NW] n1, [NW] n2
    if (lane == 0) {
        rf[warp] = s1;
        rf[NW + warp] = s2;
        ri[warp] = n1;
        ri[NW + warp] = n2;
    }
    __syncthreads();
    m1 = 0.f;
    m2 = 0.f;
    c1 = 0;
    c2 = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        m1 += rf[w];
        m2 += rf[NW + w];
        c1 += ri[w];
        c2 += ri[NW + w];
    }
    __syncthreads();
}

// Warp w's contiguous share of the units, streamed through a ring of four register
// buffers: three units' loads are in flight while one is handed to op(u, v, i) (i =
// u - u turn's first, a constant), and done(u) follows every fourth unit (units past the share are zeros, not read).  A
// unit whose largest key is at most klow is not read either (zeros).  Warp-collective.
template <bool VEC, typename Op, typename Done>
__device__ __forceinline__ void stream_units(const float* __restrict__ row, int V, int u0, int u1, const uint32_t* ukey,
                                             uint32_t klow, int lane, Op op, Done done) {
    auto load1 = [&](int u, float4* v) {
        const bool on = u < u1 && ukey[u] > klow;
#pragma unroll
        for (int j = 0; j < TB; ++j)
            v[j] = on ? load4<VEC, true>(row, V, (u * TB + j) * BLK + lane * 4, 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 R0[TB], R1[TB], R2[TB], R3[TB];
    load1(u0, R0);
    load1(u0 + 1, R1);
    load1(u0 + 2, R2);
#pragma unroll 1
    for (int u = u0; u < u1; u += 4) {
        load1(u + 3, R3);
        op(u, R0, 0);
        load1(u + 4, R0);
        op(u + 1, R1, 1);
        load1(u + 5, R1);
        op(u + 2, R2, 2);
        load1(u + 6, R2);
        op(u + 3, R3, 3);
        done(u);
    }
}

// Every run of the row that holds an element above low, appended in index order to
// warp w's slice [w * ys, (w + 1) * ys) of the second list (wn: the warp's run count;
// above ys the slice overflowed), from the row's run codes (SCAN_JOINT): (1) the code
// words of the warp's share of the units (one word per lane and unit, copied into
// shared memory first) admit the runs whose code is at least low's, and their element
// indices go in index order into the slice's index array; (2) the admitted runs are
// read through L2, 32 per lane group and eight groups in flight, and those with an
// element above low are kept in place (a kept run never moves past its own slot).  A
// unit whose largest key is at most low's admits nothing.  Warp-collective.
template <bool VEC>
__device__ __forceinline__ void compact_pass(const float* __restrict__ row, int V, int nu, float low,
                                             const uint32_t* __restrict__ code, const uint32_t* ukey, float4* y4,
                                             int* yi, int ys, int& wn, int warp, int lane) {
    int u0, u1;
    warp_range(nu, warp, u0, u1);
    float4* s4 = y4 + size_t(warp) * ys;
    int* si = yi + size_t(warp) * ys;
    const uint32_t klow = prob_key(low);
    const uint32_t clow = run_code(klow);
    const unsigned below = lanes_below(lane);
    // The code words go first into the slice's value array (free until step 2), one
    // round trip per batch of ys / 8 units.
    uint32_t* cw = reinterpret_cast<uint32_t*>(s4);
    const int ucap = ys / 8;
    int n = 0;
#pragma unroll 1
    for (int ub = u0; ub < u1; ub += ucap) {
        const int ue = min(u1, ub + ucap);
        const float* src = reinterpret_cast<const float*>(code + size_t(ub) * 32);
#pragma unroll 1
        for (int q = lane; q < (ue - ub) * 8; q += 32) cp_async16(reinterpret_cast<float*>(cw) + q * 4, src + q * 4, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll 4
        for (int u = ub; u < ue; ++u) {
            const uint32_t cur = cw[(u - ub) * 32 + lane];
            const bool on = ukey[u] > klow;
            bool adm[TB];
            unsigned bal[TB];
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                adm[j] = on && ((cur >> (8 * j)) & 0xffu) >= clow;
                bal[j] = __ballot_sync(FULL, adm[j]);
            }
            int base = n;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const int pos = base + __popc(bal[j] & below);
                if (adm[j] && pos < ys) si[pos] = ((u * TB + j) * 32 + lane) * 4;
                base += __popc(bal[j]);
            }
            n = base;
        }
        __syncwarp();
    }
    if (n > ys) {
        wn = n;
        return;
    }
    __syncwarp();
    constexpr int G = 8;  // groups of 32 admitted runs in flight
    int m = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += G * 32) {
        float4 v[G];
        int e[G];
        bool in[G];
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int c = c0 + i * 32 + lane;
            in[i] = c < n;
            e[i] = in[i] ? si[c] : 0;
            v[i] = in[i] ? load4<VEC, true>(row, V, e[i], 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncwarp();  // every lane has read its indices before any lane writes
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const bool keep = in[i] && fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)) > low;
            const unsigned bal = __ballot_sync(FULL, keep);
            const int pos = m + __popc(bal & below);
            if (keep) {
                s4[pos] = v[i];
                si[pos] = e[i];
            }
            m += __popc(bal);
        }
        __syncwarp();
    }
    wn = m;
}

// Each unit's mass above low (umass; a unit whose largest key is at most low's is 0)
// and the total in a fixed order (returned), one pass through L2; the four units' warp
// sums of a turn are interleaved.  Block-collective.
template <bool VEC>
__device__ __forceinline__ float mass_pass(const float* __restrict__ row, int V, int nu, float low, float* umass,
                                           const uint32_t* ukey, Smem sm, int warp, int lane) {
    int u0, u1;
    warp_range(nu, warp, u0, u1);
    float sm4[4];
    stream_units<VEC>(row, V, u0, u1, ukey, prob_key(low), lane,
        [&](int, const float4* v, int i) {
            float sacc = 0.f;
#pragma unroll
            for (int j = 0; j < TB; ++j)
                sacc += ((v[j].x > low ? v[j].x : 0.f) + (v[j].y > low ? v[j].y : 0.f)) +
                        ((v[j].z > low ? v[j].z : 0.f) + (v[j].w > low ? v[j].w : 0.f));
            sm4[i] = sacc;
        },
        [&](int u) {
#pragma unroll
            for (int m = 16; m; m >>= 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sm4[i] += __shfl_xor_sync(FULL, sm4[i], m);
            }
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (u + i < u1) umass[u + i] = sm4[i];
            }
        });
    __syncwarp();
    const float ws = warp_ordered_sum(umass, u0, u1, lane);
    float* rf = reinterpret_cast<float*>(sm.red()) + 24;
    if (lane == 0) rf[warp] = ws;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += rf[w];
    __syncthreads();
    return tot;
}

// The guarded locate inside chunk c of a list (one run per lane, in index order).
// Warp-collective.
__device__ __forceinline__ unsigned long long locate_in_chunk(const JList& L, const int* jb, int c, float low, float t,
                                                              int lane) {
    const int run = jb[c] + lane;
    const float4 v = L.v4[run];
    const int base = L.ix ? L.ix[run] : 4 * run;
    float rs = 0.f;
    int last_j = -1;
    float last_x = 0.f;
    unsigned long long jx = 0ull;
    if (locate_step(v, base, low, t, rs, last_j, last_x, jx, lane)) return jx;
    return pack_jx(last_j, last_x);
}

// The entry holding target t in the running sum of m[0, n) (index order), by one warp:
// lane l walks a contiguous range from the sum before it (one warp scan of the ranges'
// sums).  The first entry with positive mass whose running sum passes t, else the last
// entry with positive mass (-1 if none) ([blog] implementation details: the running sum
// is not monotone in floating point, so the pick is forced onto an eligible entry);
// `before` = the running sum before it.  Warp-collective.
__device__ __forceinline__ int locate_entry_warp(const float* m, int n, float t, int lane, float& before) {
    const int per = (n + 31) >> 5;
    const int a0 = min(n, lane * per), a1 = min(n, a0 + per);
    float own = 0.f;
#pragma unroll 4
    for (int i = a0; i < a1; ++i) own += m[i];
    const float incl = warp_incl_scan(own, lane);
    float run = incl - own;
    int hit = -1, lastpos = -1;
    float hit_before = 0.f, last_before = 0.f;
#pragma unroll 1
    for (int i = a0; i < a1; ++i) {
        const float x = m[i];
        if (x > 0.f) {
            if (hit < 0 && run + x > t) {
                hit = i;
                hit_before = run;
            }
            lastpos = i;
            last_before = run;
        }
        run += x;
    }
    const unsigned hb = __ballot_sync(FULL, hit >= 0);
    if (hb) {
        const int l = __ffs(hb) - 1;
        before = __shfl_sync(FULL, hit_before, l);
        return __shfl_sync(FULL, hit, l);
    }
    const unsigned pb = __ballot_sync(FULL, lastpos >= 0);
    if (!pb) {
        before = 0.f;
        return -1;
    }
    const int l = 31 - __clz(pb);
    before = __shfl_sync(FULL, last_before, l);
    return __shfl_sync(FULL, lastpos, l);
}

template <bool VEC>
__global__ void __launch_bounds__(NT, 1) kjoint_kernel(const SampleArgs a) {
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Smem sm(a.ns);
    const int V = a.V, ns = a.ns, nu = a.nu;
    const bool full = a.jmode != 0;
    // The row index and the parameters are read before the dependency wait (written
    // before the scan of this call started); only the summary comes from the scan.
    const int r = a.indices ? a.indices[b] : b;
    const bool row_ok = r >= 0 && r < a.batch_in;
    if (tid == NT - 32) {
        uint32_t* pr = sm.prm();
        pr[0] = uint32_t(a.top_k ? a.top_k[b] : 0);
        pr[1] = __float_as_uint(a.top_p ? a.top_p[b] : 1.f);
        pr[2] = __float_as_uint(a.min_p ? a.min_p[b] : 0.f);
        *reinterpret_cast<unsigned long long*>(pr + 4) = a.seeds ? a.seeds[b] : a.seed;
    }
    if (!full)
        for (int i = tid; i < HBINS; i += NT) sm.hist()[i] = 0u;
    const float* row = a.probs + size_t(row_ok ? r : 0) * size_t(V);
    if (full && row_ok) {
        // The whole row into shared memory (its blocks become the chunks), issued before
        // the wait: the input rows were written before the scan of this call started.
        float* stg = sm.at<float>(jx_off(ns));
#pragma unroll 1
        for (int c = warp; c < ns; c += NW) stage4<VEC>(stg + c * BLK + lane * 4, row, V, c * BLK + lane * 4);
        cp_async_commit();
    }
    grid_dependency_wait();
    allow_dependents();
    if (b == 0 && tid < SCAN_CTRS && a.sctr) a.sctr[tid * SCAN_CTR_STRIDE] = 0u;  // the scan is complete
    if (tid == NT - 32) {  // a device-resident offset may be advanced by the kernel before
        *reinterpret_cast<unsigned long long*>(sm.prm() + 6) =
            (a.offsets ? a.offsets[b] : a.offset) + (a.offset_dev ? *a.offset_dev : 0ull);
    }
    float* umass = sm.mass(1);
    uint32_t* ukey = reinterpret_cast<uint32_t*>(sm.mass(2));
    // ---- the summary: in jmode 1 with the segment masses (the first draw's table), in
    // jmode 0 with the unit masses and keys and the histogram of the block maxima
    if (row_ok) {
        if (full)
            load_summary(a, r, sm, true, warp, lane, tid);
        else
            load_summary(a, r, sm, false, warp, lane, tid, nullptr, umass, ukey, sm.hist());
    } else {
        __syncthreads();
    }
    const int k = int(sm.prm()[0]);
    const bool k_on = k > 0 && k < V;
    const float mp_row = __uint_as_float(sm.prm()[2]);
    const bool m_on = mp_row > 0.f;  // a min-p filter: f fails below min_p * max
    // jmode 0 needs a threshold below which f fails: the top-k bound (ns >= k) or min-p
    if (!row_ok || a.shift != 0 || (!full && !(k_on && ns >= k) && !m_on)) {
        cp_async_wait<0>();
        __syncthreads();
        sample_row_fin<VEC>(a);
        return;
    }
    const unsigned long long seed_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 4);
    const unsigned long long offset_b = *reinterpret_cast<const unsigned long long*>(sm.prm() + 6);
    const uint32_t stream_b = a.seeds ? 0u : uint32_t(b);
    float* uni = reinterpret_cast<float*>(sm.red()) + (REDW - 32);  // [32] the uniforms of rounds 0..31
    if (warp == NW - 1) uni[lane] = sampler_uniform(seed_b, offset_b, stream_b, uint32_t(lane));
    float* jm0 = sm.at<float>(jtab_off(ns));
    float* jm1 = jm0 + JCH;
    int* jb = reinterpret_cast<int*>(jm0 + 2 * JCH);
    float* jk = jm0 + 3 * JCH;
    JList L;
    const float* cur = nullptr;  // each chunk's mass above low, while low >= L.lo
    float4* y4 = nullptr;
    int* yi = nullptr;
    const int ys = a.jy4 / NW;  // runs per warp slice of the second list (a multiple of 32)
    if (full) {
        float4* v4 = sm.at<float4>(jx_off(ns));
        for (int c = tid; c < ns; c += NT) {
            jb[c] = 32 * c;
            jk[c] = __uint_as_float(sm.segkey()[c]);
        }
        cp_async_wait<0>();
        __syncthreads();
        L.v4 = v4;
        L.ix = nullptr;
        L.nch = ns;
        L.lo = 0.f;
        cur = sm.mass(0);
    } else {
        // ---- the first draw, by warp 0 while the others build the candidate list: over
        // the whole row (low = 0), from the scan's unit masses and one read of the unit.
        // It is used when the first round runs below the list's threshold (uk > 1).
        if (warp == 0) {
            const float t = sampler_uniform(seed_b, offset_b, stream_b, 0u) * sm.part()[0].f[0];
            float before = 0.f;
            const int un = locate_entry_warp(umass, nu, t, lane, before);
            unsigned long long jx = pack_jx(-1, 0.f);
            if (un >= 0) jx = locate_in_unit<VEC>(row, V, un, 0.f, fmaxf(t - before, 0.f), lane);
            if (lane == 0) {
                sm.red()[88] = unpack_j(jx);
                reinterpret_cast<float*>(sm.red())[92] = unpack_x(jx);
            }
        }
        // ---- uk; the live blocks (largest value >= uk) copied in index order into the
        // second list's area (one round trip to L2), then each warp appends the runs of its
        // own live blocks that hold a candidate
        const bool kb = k_on && ns >= k;  // the top-k bound is available
        if (warp == 1 && kb) {
            uint32_t above;
            const int B = scan_bins_down<uint32_t>(sm.hist(), int(min(uint32_t(HBINS - 1), sm.part()[0].u[2] >> 21)),
                                                   uint32_t(k), lane, above);
            if (lane == 0) sm.bcast()[0] = max(B, 0);
        }
        __syncthreads();
        // uk: the larger of the top-k bound and the min-p threshold (the float32 of
        // min_p * max rounded up, as f takes it), below either of which f fails.
        const uint32_t uk_k = kb ? max(1u, uint32_t(sm.bcast()[0]) << 21) : 0u;
        const uint32_t uk_m =
            m_on ? prob_key(__double2float_ru(double(mp_row) * double(__uint_as_float(sm.part()[0].u[2])))) : 0u;
        const uint32_t uk = max(1u, max(uk_k, uk_m));  // zeros are never candidates
        const bool by_min_p = m_on && uk_m >= uk_k;     // f fails below uk by min-p, whatever the count
        const float lo = __uint_as_float(uk - 1u);      // x > lo  <=>  x >= the float of uk
        int r0, r1;
        warp_range(ns, warp, r0, r1);
        int nl = 0;
#pragma unroll 1
        for (int b0 = r0; b0 < r1; b0 += 32)
            nl += __popc(__ballot_sync(FULL, b0 + lane < r1 && sm.segkey()[b0 + lane] >= uk));
        if (lane == 0) sm.red()[warp] = nl;
        __syncthreads();
        int off = 0, nlive = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int c = sm.red()[w];
            off += w < warp ? c : 0;
            nlive += c;
        }
        const int yblocks = int((size_t(a.jy4) * 20) / (BLK * 4));
        if (nlive > yblocks) {
            __syncthreads();
            sample_row_fin<VEC>(a);
            return;
        }
        float* stg = sm.at<float>(jy_off(ns));
        int* seg = sm.list();  // [nlive] the staged blocks, in index order
        const int off0 = off;
#pragma unroll 1
        for (int b0 = r0; b0 < r1; b0 += 32) {
            unsigned bal = __ballot_sync(FULL, b0 + lane < r1 && sm.segkey()[b0 + lane] >= uk);
#pragma unroll 1
            while (bal) {
                const int sg = b0 + __ffs(bal) - 1;
                bal &= bal - 1u;
                stage4<VEC>(stg + off * BLK + lane * 4, row, V, sg * BLK + lane * 4);
                if (lane == 0) seg[off] = sg;
                ++off;
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();  // every warp's copies and block numbers
        float4* x4 = sm.at<float4>(jx_off(ns));
        int* xi = sm.at<int>(jx_off(ns) + size_t(JX4) * 16);
        constexpr int XS = JX4 / NW;
        int wn = 0, cnt = 0;
        const float4* stg4 = reinterpret_cast<const float4*>(stg);
#pragma unroll 1
        for (int q = off0; q < off0 + nl; ++q) {
            const float4 v = stg4[q * 32 + lane];
            append_run(v, seg[q] * BLK + lane * 4, lo, x4 + warp * XS, xi + warp * XS, XS, wn, lane);
            cnt += int(v.x > lo) + int(v.y > lo) + int(v.z > lo) + int(v.w > lo);
        }
        cnt = warp_sum_i(cnt);
        if (lane == 0) sm.red()[warp] = cnt;  // words 0 .. NW: no other use after the summary
        const int nch = close_list(x4, XS, wn, jb, jk, sm, warp, lane);  // its barriers publish the counts
        int n = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) n += sm.red()[w];
        if (nch < 0 || (!by_min_p && n < k)) {
            __syncthreads();
            sample_row_fin<VEC>(a);
            return;
        }
        L.v4 = x4;
        L.ix = xi;
        L.nch = nch;
        L.lo = lo;
        y4 = sm.at<float4>(jy_off(ns));
        yi = sm.at<int>(jy_off(ns) + size_t(a.jy4) * 16);
    }
    // ---- the rounds ([blog] dual-pivot rejection sampling)
    const float tp = __uint_as_float(sm.prm()[1]);
    const float mp = __uint_as_float(sm.prm()[2]);
    const float M = sm.part()[0].f[0];
    const bool any_bad = sm.part()[0].u[1] != 0u;
    const float rowmax = __uint_as_float(sm.part()[0].u[2]);
    Pred f;
    f.single = a.single_pivot != 0;
    f.k_on = k_on;
    f.k = k;
    f.p_on = tp < 1.f;
    f.m_on = mp > 0.f;
    f.pthr = tp * M;
    f.t32 = 0.f;
    bool valid = !isnan(tp) && !isnan(mp) && !any_bad && M > 0.f && M <= 3.402823466e38f;
    if (f.m_on) {
        f.t32 = __double2float_ru(double(mp) * double(rowmax));
        if (!(rowmax >= f.t32)) valid = false;
    }
    int* st = sm.red() + 88;                               // [4] round results (ints)
    float* sf = reinterpret_cast<float*>(sm.red()) + 92;  // [4] round results (floats)
    float low = 0.f, high = rowmax, S_low = M;
    if (!full && L.lo <= 0.f) {  // every positive element is a candidate: the list serves from the first draw
        float m2 = 0.f;
        int c1 = 0, c2 = 0;
        chunk_pass(L, jb, jk, 0.f, 0.f, jm0, jm1, sm, tid, warp, lane, S_low, m2, c1, c2);
        cur = jm0;
    }
    int token = -1, rounds = 0;
#pragma unroll 1
    for (int round = 0; valid && round < R_MAX; ++round) {
        const float u = round < 32 ? uni[round] : sampler_uniform(seed_b, offset_b, stream_b, uint32_t(round));
        // ---- below the list's threshold after the first round: one pass through L2 copies
        // every run above low into the second list, whose chunk masses above low are then
        // this draw's table; if that list overflows, the pass gives each unit's mass above low
        if (low < L.lo && round > 0) {
            int nch = -1;
            if (ys >= 32) {
                int wn = 0;
                compact_pass<VEC>(row, V, nu, low, a.scode + size_t(r) * nu * 32, ukey, y4, yi, ys, wn, warp, lane);
                nch = close_list(y4, ys, wn, jb, jk, sm, warp, lane);
            }
            if (nch >= 0) {
                L.v4 = y4;
                L.ix = yi;
                L.nch = nch;
                L.lo = low;
                float m2 = 0.f;
                int c1 = 0, c2 = 0;
                chunk_pass(L, jb, jk, low, low, jm0, jm1, sm, tid, warp, lane, S_low, m2, c1, c2);
                cur = jm0;
            } else {
                S_low = mass_pass<VEC>(row, V, nu, low, umass, ukey, sm, warp, lane);
            }
        }
        // ---- draw j by inverse transform over the tokens above low ([blog]): from the
        // list's chunk masses, else from the unit masses and the unit read through L2 (the
        // first round's below-threshold draw was made during the set-up)
        if (warp == 0 && !(round == 0 && low < L.lo)) {
            const float t = u * S_low;
            float before = 0.f;
            unsigned long long jx = pack_jx(-1, 0.f);
            if (low >= L.lo) {
                const int c = locate_entry_warp(cur, L.nch, t, lane, before);
                if (c >= 0) jx = locate_in_chunk(L, jb, c, low, fmaxf(t - before, 0.f), lane);
            } else {
                const int un = locate_entry_warp(umass, nu, t, lane, before);
                if (un >= 0) jx = locate_in_unit<VEC>(row, V, un, low, fmaxf(t - before, 0.f), lane);
            }
            if (lane == 0) {
                st[0] = unpack_j(jx);
                sf[0] = unpack_x(jx);
            }
        }
        __syncthreads();
        const int j = st[0];
        const float pivot1 = sf[0];
        if (j < 0) break;
        const float pivot2 = f.pivot2(pivot1, high);
        // ---- f at both pivots: from the list at or above its threshold, else false
        int kase = 3;
        float m1 = 0.f, m2 = 0.f;
        if (fmaxf(pivot1, pivot2) >= L.lo) {
            int c1 = 0, c2 = 0;
            chunk_pass(L, jb, jk, pivot1, pivot2, jm0, jm1, sm, tid, warp, lane, m1, m2, c1, c2);
            const bool f1 = pivot1 >= L.lo && f(c1, m1, pivot1);
            const bool f2 = pivot2 >= L.lo && f(c2, m2, pivot2);
            kase = f1 ? 1 : (f2 ? 2 : 3);
        }
        if (kase == 1) {
            token = j;
            rounds = round + 1;
            break;
        }
        if (kase == 2) {
            low = pivot1;
            high = pivot2;
            S_low = m1;
            cur = jm0;
        } else {
            low = pivot2;
            S_low = m2;
            cur = jm1;
        }
        if (round == R_MAX - 1) rounds = R_MAX;
    }
    if (tid == 0) {
        a.out_token[b] = token >= 0 ? token : -1;
        a.out_valid[b] = token >= 0 ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = token >= 0 ? rounds : (valid ? R_MAX : 0);
    }
}

// ------------------------------------------------------------------ lean draw (no filter)
//
// The finishing launch of sampling without filters on rows of probabilities, one warp
// per output row.  With no filter f holds at every pivot, so the first draw of the
// rejection sampler is the sample ([blog] dual-pivot rejection sampling: accept j when
// f(p_j) holds): the inverse transform over the whole row ([blog] inverse transform
// sampling), from the scan's unit masses (lane l sums a contiguous range of units; one
// warp scan gives M and every range's start), the guarded pick of the unit, then the
// element inside the unit read through L2.  Two round trips to L2 after the scan.
template <bool VEC>
__global__ void __launch_bounds__(NT) kdraw_kernel(const SampleArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = int(blockIdx.x) * NW + warp;
    const bool in_range = b < a.nout;
    // Read before the dependency wait: written before the scan of this call started.
    const int r = in_range ? (a.indices ? a.indices[b] : b) : -1;
    const unsigned long long seed_b = in_range ? (a.seeds ? a.seeds[b] : a.seed) : 0ull;
    grid_dependency_wait();
    allow_dependents();
    if (b == 0 && lane < SCAN_CTRS && a.sctr) a.sctr[lane * SCAN_CTR_STRIDE] = 0u;  // the scan is complete
    if (!in_range) return;
    const unsigned long long offset_b =
        (a.offsets ? a.offsets[b] : a.offset) + (a.offset_dev ? *a.offset_dev : 0ull);
    const uint32_t stream_b = a.seeds ? 0u : uint32_t(b);
    const int nu = a.nu;
    int token = -1;
    bool valid = false;
    if (r >= 0 && r < a.batch_in) {
        const uint4* st = a.sstat + size_t(r) * nu;
        const int per = (nu + 31) >> 5;
        const int a0 = min(nu, lane * per), a1 = min(nu, a0 + per);
        // The lane's unit masses in registers (KD units at a time, every load issued
        // before the first is used); ranges longer than KD are read again for the walk.
        constexpr int KD = 16;
        float um[KD];
        float own = 0.f;
        bool bad = false;
#pragma unroll 1
        for (int c0 = a0; c0 < a1; c0 += KD) {
#pragma unroll
            for (int q = 0; q < KD; ++q) {
                const uint4 v = c0 + q < a1 ? __ldcg(st + c0 + q) : make_uint4(0u, 0u, 0u, 0u);
                um[q] = __uint_as_float(v.x);
                bad |= v.z != 0u;
            }
#pragma unroll
            for (int q = 0; q < KD; ++q) own += um[q];
        }
        const float incl = warp_incl_scan(own, lane);
        const float M = __shfl_sync(FULL, incl, 31);
        bad = __any_sync(FULL, bad);
        valid = !bad && M > 0.f && M <= 3.402823466e38f;
        if (valid) {
            const float t = sampler_uniform(seed_b, offset_b, stream_b, 0u) * M;
            // the first unit with positive mass whose running sum passes t, else the last
            // unit with positive mass (the sum is not monotone in floating point)
            float run = incl - own;
            int hit = -1, lastpos = -1;
            float hit_before = 0.f, last_before = 0.f;
            const bool in_regs = a1 - a0 <= KD;
#pragma unroll 1
            for (int c0 = a0; c0 < a1; c0 += KD) {
                if (!in_regs) {
#pragma unroll
                    for (int q = 0; q < KD; ++q) um[q] = c0 + q < a1 ? __uint_as_float(__ldcg(&st[c0 + q].x)) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < KD; ++q) {
                    const float m = um[q];
                    if (c0 + q < a1 && m > 0.f) {
                        if (hit < 0 && run + m > t) {
                            hit = c0 + q;
                            hit_before = run;
                        }
                        lastpos = c0 + q;
                        last_before = run;
                    }
                    run += m;
                }
            }
            const unsigned hb = __ballot_sync(FULL, hit >= 0);
            const unsigned pb = __ballot_sync(FULL, lastpos >= 0);
            int un = -1;
            float before = 0.f;
            if (hb) {
                const int l = __ffs(hb) - 1;
                un = __shfl_sync(FULL, hit, l);
                before = __shfl_sync(FULL, hit_before, l);
            } else if (pb) {
                const int l = 31 - __clz(pb);
                un = __shfl_sync(FULL, lastpos, l);
                before = __shfl_sync(FULL, last_before, l);
            }
            if (un >= 0) {
                const float* row = a.probs + size_t(r) * size_t(a.V);
                token = unpack_j(locate_in_unit<VEC>(row, a.V, un, 0.f, fmaxf(t - before, 0.f), lane));
            }
        }
    }
    if (lane == 0) {
        a.out_token[b] = token >= 0 ? token : -1;
        a.out_valid[b] = token >= 0 ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = token >= 0 ? 1 : (valid ? R_MAX : 0);
    }
}

// ------------------------------------------------------------------ host side

#ifndef FS_SCAN_PER_SM
#define FS_SCAN_PER_SM 4   // scan CTAs per SM (the occupancy of scan_kernel: every SM gets as many)
#endif

// Grid of the scan: one wave of FS_SCAN_PER_SM CTAs per SM, fewer when the matrix has
// fewer units than the wave has warps.
static fs_status scan_grid(long long units, int& grid) {
    int sms = 0;
    size_t optin = 0;
    const fs_status st = device_limits(sms, optin);
    if (st != FS_OK) return st;
    const long long want = (units + NW - 1) / NW;
    const long long wave = (long long)sms * FS_SCAN_PER_SM;
    grid = int(want < wave ? want : wave);
    return FS_OK;
}

template <int KIND>
static fs_status launch_scan(const float* x, int rows, int V, int shift, int ns, bool vec, void* ws, void* stream) {
    ScanArgs s;
    s.x = x;
    s.rows = rows;
    s.V = V;
    s.shift = shift;
    s.ns = ns;
    s.nu = scan_units(V);
    s.ls = scan_row_words(ns);
    char* body = reinterpret_cast<char*>(ws) + SCAN_HEAD;
    s.key = reinterpret_cast<uint32_t*>(body);
    s.mass = reinterpret_cast<float*>(body + size_t(rows) * s.ls * 4);
    s.stat = reinterpret_cast<uint4*>(body + 2 * size_t(rows) * s.ls * 4);
    s.code = reinterpret_cast<uint32_t*>(body + 2 * size_t(rows) * s.ls * 4 + size_t(rows) * s.nu * 16);
    s.ctr = reinterpret_cast<unsigned*>(ws);
    const long long total = (long long)rows * s.nu;
    s.ustatic = total - total / 5;
    s.slice = int((total - s.ustatic + SCAN_CTRS - 1) / SCAN_CTRS);
    int grid = 0;
    fs_status st = scan_grid(total, grid);
    if (st != FS_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = vec ? cudaLaunchKernelEx(&cfg, scan_kernel<true, KIND>, s)
                        : cudaLaunchKernelEx(&cfg, scan_kernel<false, KIND>, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return FS_OK;
}

// The scan of the input rows, then the finishing launch (one CTA per output row).
static fs_status launch_scan_finish(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                    int32_t batch_out, const int32_t* top_k, const float* top_p, const float* min_p,
                                    int32_t order, uint64_t seed, uint64_t offset, int32_t* out_token,
                                    uint8_t* out_valid, int32_t* out_rounds, void* stream, const uint64_t* seeds,
                                    const uint64_t* offsets, const uint64_t* offset_dev, int32_t pivots, bool soft,
                                    const float* temperature, bool vec, void* fixed_ws = nullptr) {
    const bool kfirst = order == FS_ORDER_TOP_K_FIRST && top_k;
    const bool kjoint = !soft && order == FS_ORDER_JOINT && (top_k || min_p);
    const bool kdraw = !soft && !top_k && !top_p && !min_p;  // no filter: the first draw is the sample
    auto fin_fn = [&]() -> void (*)(SampleArgs) {
        if (soft) return vec ? sample_kernel<true, true, true> : sample_kernel<false, true, true>;
        if (kfirst) return vec ? kfirst_kernel<true> : kfirst_kernel<false>;
        if (kjoint) return vec ? kjoint_kernel<true> : kjoint_kernel<false>;
        if (kdraw) return vec ? kdraw_kernel<true> : kdraw_kernel<false>;
        return vec ? sample_kernel<true, false, true> : sample_kernel<false, false, true>;
    };
    void (*fn)(SampleArgs) = fin_fn();
    fs_status st = prepare_kernel(reinterpret_cast<const void*>(fn));
    if (st != FS_OK) return st;
    int sms = 0;
    size_t optin = 0;
    st = device_limits(sms, optin);
    if (st != FS_OK) return st;
    Plan p;
    p.C = 1;
    p.shift = seg_shift_for(vocab);
    p.ns = (vocab + (BLK << p.shift) - 1) / (BLK << p.shift);
    p.nsc = (p.ns + 3) & ~3;
    p.smem = (kfirst && !soft) ? kfirst_smem(p.ns) : Layout(p.ns).total();
    int jmode = 0, jy4 = 0;
    if (kjoint) {
        // The whole row when it fits beside the tables; else the candidate list and, in
        // the rest of the device's limit, the second list (whole chunks per warp).
        const size_t row_end = jx_off(p.ns) + size_t(p.ns) * BLK * 4;
        if (p.shift == 0 && p.ns <= JCH && row_end <= optin) {
            jmode = 1;
            p.smem = row_end;
        } else {
            p.smem = optin;
            if (optin > jy_off(p.ns)) {
                constexpr size_t quantum = size_t(NW) * 32;
                jy4 = int((optin - jy_off(p.ns)) / 20 / quantum * quantum);
                if (jy4 > JCH * 32) jy4 = JCH * 32;  // its chunks fit the table
            }
        }
    }
    p.per_sm = 0;
    if (p.smem > optin || (kjoint && p.smem < jy_off(p.ns) && jmode == 0)) return FS_ERR_UNSUPPORTED;
    void* ws = nullptr;
    // Top-k-first launches draw from gathered candidates and unfiltered ones from the unit
    // records: no segment masses needed.
    if (batch_in > 0) {
        if (fixed_ws) {
            ws = fixed_ws;  // caller-checked to hold the summaries
        } else {
            st = workspace(scan_workspace_bytes(batch_in, vocab, kjoint), stream, &ws);
            if (st != FS_OK) return st;
        }
        if (soft)
            st = launch_scan<SCAN_LOGITS>(probs, batch_in, vocab, p.shift, p.ns, vec, ws, stream);
        else if (kfirst || kdraw)  // kdraw reads only the unit records
            st = launch_scan<SCAN_KEYS>(probs, batch_in, vocab, p.shift, p.ns, vec, ws, stream);
        else if (kjoint)
            st = launch_scan<SCAN_JOINT>(probs, batch_in, vocab, p.shift, p.ns, vec, ws, stream);
        else
            st = launch_scan<SCAN_MASSES>(probs, batch_in, vocab, p.shift, p.ns, vec, ws, stream);
        if (st != FS_OK) return st;
    }
    SampleArgs a = {};
    a.probs = probs;
    a.batch_in = batch_in;
    a.V = vocab;
    a.indices = indices;
    a.top_k = top_k;
    a.top_p = top_p;
    a.min_p = min_p;
    a.order = order == FS_ORDER_TOP_K_FIRST ? 0 : 1;
    a.seed = seed;
    a.offset = offset;
    a.seeds = reinterpret_cast<const unsigned long long*>(seeds);
    a.offsets = reinterpret_cast<const unsigned long long*>(offsets);
    a.offset_dev = reinterpret_cast<const unsigned long long*>(offset_dev);
    a.single_pivot = pivots == 1 ? 1 : 0;
    a.temperature = temperature;
    a.out_token = out_token;
    a.out_valid = out_valid;
    a.out_rounds = out_rounds;
    a.shift = p.shift;
    a.ns = p.ns;
    a.nsc = p.nsc;
    a.ls = scan_row_words(p.ns);
    a.nu = scan_units(vocab);
    const char* body = ws ? reinterpret_cast<const char*>(ws) + SCAN_HEAD : nullptr;
    a.skey = ws ? reinterpret_cast<const uint32_t*>(body) : nullptr;
    a.smass = (ws && !soft && !kfirst && !kdraw) ? reinterpret_cast<const float*>(body + size_t(batch_in) * a.ls * 4)
                                                 : nullptr;  // the joint order: segment masses
    a.sstat = ws ? reinterpret_cast<const uint4*>(body + 2 * size_t(batch_in) * a.ls * 4) : nullptr;
    a.scode = (ws && kjoint) ? reinterpret_cast<const uint32_t*>(body + 2 * size_t(batch_in) * a.ls * 4 +
                                                                  size_t(batch_in) * a.nu * 16)
                             : nullptr;
    a.sctr = reinterpret_cast<unsigned*>(ws);
    a.jmode = jmode;
    a.jy4 = jy4;
    a.nout = batch_out;
    if (kdraw) {  // one warp per output row, no shared memory
        p.smem = 0;
        return launch_cluster(fn, p, (batch_out + NW - 1) / NW, stream, a);
    }
    return launch_cluster(fn, p, batch_out, stream, a);
}

static fs_status launch_sample(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                               int32_t batch_out, const int32_t* top_k, const float* top_p, const float* min_p,
                               int32_t order, uint64_t seed, uint64_t offset, int32_t* out_token, uint8_t* out_valid,
                               int32_t* out_rounds, void* stream, const uint64_t* seeds = nullptr,
                               const uint64_t* offsets = nullptr, const uint64_t* offset_dev = nullptr,
                               int32_t pivots = 2, bool soft = false, const float* temperature = nullptr,
                               void* fixed_ws = nullptr) {
    if (batch_out < 0 || batch_in < 0) return FS_ERR_INVALID_ARG;
    if (batch_out == 0) return FS_OK;
    if (!probs || !out_token || !out_valid) return FS_ERR_INVALID_ARG;
    if (vocab < 1) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    if (!indices && batch_out != batch_in) return FS_ERR_INVALID_ARG;
    if (order != FS_ORDER_TOP_K_FIRST && order != FS_ORDER_JOINT) return FS_ERR_INVALID_ARG;
    if (pivots != 1 && pivots != 2) return FS_ERR_INVALID_ARG;

    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(probs) & 15) == 0);
    // One streaming pass per row: the top-k-first order, and sampling without filters.
    const bool single_pass = (order == FS_ORDER_TOP_K_FIRST && top_k) || (!top_k && !top_p && !min_p);
    // Those run as a scan of the input rows and a finishing launch per output row
    // (masses of logits depend on the temperature, so sampling logits without filters
    // stays on the clusters).
    const bool fin = (order == FS_ORDER_TOP_K_FIRST && top_k) || (!soft && !top_k && !top_p && !min_p) ||
                     (!soft && order == FS_ORDER_JOINT && (top_k || min_p));
    if (fin) return launch_scan_finish(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed,
                                       offset, out_token, out_valid, out_rounds, stream, seeds, offsets, offset_dev,
                                       pivots, soft, temperature, vec, fixed_ws);
    const void* fn = soft ? (vec ? reinterpret_cast<const void*>(sample_kernel<true, true, false>)
                                 : reinterpret_cast<const void*>(sample_kernel<false, true, false>))
                          : (vec ? reinterpret_cast<const void*>(sample_kernel<true, false, false>)
                                 : reinterpret_cast<const void*>(sample_kernel<false, false, false>));
    Plan p;
    fs_status st = make_plan(batch_out, vocab, fn, single_pass, p);
    if (st != FS_OK) return st;
    SampleArgs a = {};
    a.probs = probs;
    a.batch_in = batch_in;
    a.V = vocab;
    a.indices = indices;
    a.top_k = top_k;
    a.top_p = top_p;
    a.min_p = min_p;
    a.order = order == FS_ORDER_TOP_K_FIRST ? 0 : 1;
    a.seed = seed;
    a.offset = offset;
    a.seeds = reinterpret_cast<const unsigned long long*>(seeds);
    a.offsets = reinterpret_cast<const unsigned long long*>(offsets);
    a.offset_dev = reinterpret_cast<const unsigned long long*>(offset_dev);
    a.single_pivot = pivots == 1 ? 1 : 0;
    a.temperature = temperature;
    a.out_token = out_token;
    a.out_valid = out_valid;
    a.out_rounds = out_rounds;
    a.shift = p.shift;
    a.ns = p.ns;
    a.nsc = p.nsc;
    if (soft) {
        if (vec) return launch_cluster(sample_kernel<true, true, false>, p, batch_out, stream, a);
        return launch_cluster(sample_kernel<false, true, false>, p, batch_out, stream, a);
    }
    if (vec) return launch_cluster(sample_kernel<true, false, false>, p, batch_out, stream, a);
    return launch_cluster(sample_kernel<false, false, false>, p, batch_out, stream, a);
}

// ------------------------------------------------------------------ scratch without allocation
//
// For callers that may not allocate device memory: fs_top_k_top_p_sampling_noalloc keeps
// the row summaries of its scan in this fixed array instead of the per-stream buffers.
// It is part of the module image, so every device that loads the library holds it until
// the process exits.  Host code cannot pass the array's name to a kernel (on the host
// it names a stand-in, not device memory): its device address is looked up once per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FS_NOALLOC_SCRATCH_BYTES];

static fs_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return FS_ERR_UNSUPPORTED;
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        addr[dev] = p;
    }
    *out = addr[dev];
    return FS_OK;
}

__global__ void advance_kernel(unsigned long long* offset_dev, unsigned long long delta) {
    grid_dependency_wait();
    *offset_dev += delta;
}

}  // namespace fsd

extern "C" {

fs_status fs_sampling_from_probs(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                 int32_t batch_out, uint64_t seed, uint64_t offset, int32_t* out_token,
                                 uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, nullptr, nullptr, FS_ORDER_JOINT,
                              seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_k_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const int32_t* top_k, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!top_k && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, nullptr, nullptr, FS_ORDER_JOINT,
                              seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const float* top_p, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!top_p && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, top_p, nullptr, FS_ORDER_JOINT,
                              seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_min_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const float* min_p, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!min_p && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, nullptr, min_p, FS_ORDER_JOINT,
                              seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_k_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                  int32_t batch_out, const int32_t* top_k, const float* top_p, const float* min_p,
                                  int32_t order, uint64_t seed, uint64_t offset, int32_t* out_token,
                                  uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if ((!top_k || !top_p) && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed, offset,
                              out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_k_top_p_sampling_noalloc(const float* probs, int32_t batch_in, int32_t vocab,
                                          const int32_t* indices, int32_t batch_out, const int32_t* top_k,
                                          const float* top_p, const float* min_p, int32_t order, uint64_t seed,
                                          uint64_t offset, int32_t* out_token, uint8_t* out_valid,
                                          int32_t* out_rounds, void* stream) {
    if ((!top_k || !top_p) && batch_out > 0) return FS_ERR_INVALID_ARG;
    void* scratch = nullptr;
    // Both orders run as the scan and a finishing launch here (top_k is given); the joint
    // order's summaries also hold the run codes.
    if (batch_out > 0 && batch_in > 0 && vocab >= 1 && vocab <= FS_MAX_VOCAB) {
        const size_t need = fsd::scan_workspace_bytes(batch_in, vocab, order == FS_ORDER_JOINT);
        if (need > size_t(FS_NOALLOC_SCRATCH_BYTES)) {
            fsd::set_last_error("fs_top_k_top_p_sampling_noalloc: the row summaries of this batch need more than "
                                "FS_NOALLOC_SCRATCH_BYTES of fixed scratch (see fs_workspace_bytes)");
            return FS_ERR_UNSUPPORTED;
        }
        const fs_status st = fsd::noalloc_scratch(&scratch);
        if (st != FS_OK) return st;
        // The scan's claim counters (the first words of its scratch) start at zero.
        const cudaError_t e = cudaMemsetAsync(scratch, 0, fsd::SCAN_HEAD, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fsd::cuda_fail(e);
    }
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed, offset,
                              out_token, out_valid, out_rounds, stream, nullptr, nullptr, nullptr, 2, false, nullptr,
                              scratch);
}

fs_status fs_top_k_top_p_sampling_rng(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                      int32_t batch_out, const int32_t* top_k, const float* top_p, const float* min_p,
                                      int32_t order, const uint64_t* seeds, const uint64_t* offsets,
                                      const uint64_t* offset_dev, uint64_t seed, uint64_t offset, int32_t* out_token,
                                      uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed, offset,
                              out_token, out_valid, out_rounds, stream, seeds, offsets, offset_dev);
}

fs_status fs_advance_offset(uint64_t* offset_dev, uint64_t delta, void* stream) {
    if (!offset_dev) return FS_ERR_INVALID_ARG;
    fsd::advance_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<unsigned long long*>(offset_dev), static_cast<unsigned long long>(delta));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fsd::cuda_fail(e);
    return FS_OK;
}

fs_status fs_top_k_top_p_sampling_pivots(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                         int32_t batch_out, const int32_t* top_k, const float* top_p,
                                         const float* min_p, int32_t order, int32_t pivots, uint64_t seed,
                                         uint64_t offset, int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds,
                                         void* stream) {
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed, offset,
                              out_token, out_valid, out_rounds, stream, nullptr, nullptr, nullptr, pivots);
}

fs_status fs_top_k_top_p_sampling_from_logits(const float* logits, int32_t batch_in, int32_t vocab,
                                              const int32_t* indices, int32_t batch_out, const float* temperature,
                                              const int32_t* top_k, const float* top_p, const float* min_p,
                                              int32_t order, uint64_t seed, uint64_t offset, int32_t* out_token,
                                              uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    return fsd::launch_sample(logits, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed, offset,
                              out_token, out_valid, out_rounds, stream, nullptr, nullptr, nullptr, 2, true,
                              temperature);
}

fs_status fs_sampling_plan(int32_t batch_out, int32_t vocab, int32_t order, int32_t* cluster,
                           int32_t* segment_len, int32_t* segments_per_cta, int32_t* ctas_per_sm) {
    if (batch_out < 1 || vocab < 1 || !cluster || !segment_len || !segments_per_cta || !ctas_per_sm)
        return FS_ERR_INVALID_ARG;
    if (order != FS_ORDER_TOP_K_FIRST && order != FS_ORDER_JOINT) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    if (order == FS_ORDER_TOP_K_FIRST) {
        // The scan and the finishing launch: one CTA per row finishes it from the whole
        // row's summary; the scan keeps FS_SCAN_PER_SM CTAs on every SM.
        const int shift = fsd::seg_shift_for(vocab);
        *cluster = 1;
        *segment_len = fsd::BLK << shift;
        *segments_per_cta = (vocab + (fsd::BLK << shift) - 1) / (fsd::BLK << shift);
        *ctas_per_sm = FS_SCAN_PER_SM;
        return FS_OK;
    }
    // Clusters: the plan of rows of probabilities that are 16-byte aligned with V % 4 = 0
    // (the other rows run a scalar-load build of the same kernel, whose occupancy can
    // differ).
    fsd::Plan p;
    const fs_status st = fsd::make_plan(batch_out, vocab, reinterpret_cast<const void*>(fsd::sample_kernel<true, false, false>),
                                       false, p);
    if (st != FS_OK) return st;
    *cluster = p.C;
    *segment_len = fsd::BLK << p.shift;
    *segments_per_cta = p.nsc;
    *ctas_per_sm = p.per_sm;
    return FS_OK;
}

}  // extern "C"
