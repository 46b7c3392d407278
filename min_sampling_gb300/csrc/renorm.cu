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
//            top-p: bisection on the key with three pivots per pass, each interval
//            shrunk to the keys that exist in it;
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

// Write this CTA's segments: keep key >= t (x / denom, or the logit), else fill.
// Segments whose maximum key is below t are written without being read.
template <bool VEC, int KIND>
__device__ __forceinline__ void write_pass(const float* __restrict__ row, float* __restrict__ orow, Geom g,
                                       Smem sm, bool valid, uint32_t t, float denom, int warp, int lane) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyLogit, KeyProb>::type;
    constexpr bool IS_PROB = KIND != K_MASK;
    const KEYF keyf;
    const float fill = IS_PROB ? 0.f : __int_as_float(0xff800000);
    const bool vec_out = VEC && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
    stream_warp<VEC, false>(
        row, g, sm, warp, lane, [&](int sg) { return valid && sm.segkey()[sg] >= t; },
        [&](int, int, bool on, const float4& v, int base) {
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

template <bool VEC, int KIND>
__global__ void __launch_bounds__(NT, 4) filter_kernel(const FilterArgs a) {
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
                 lane, tid);
    cluster_sync();  // the leader's segment table, every CTA's parts and histogram, are complete

    const Totals tot = cluster_totals(sm, C);
    const int npos = tot.npos;
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
    if (k_on) {
        L0 = need_hist ? hist_bound(sm, g, rank, C, k, maxkey, warp, lane, tid) : 0u;
        if (IS_PROB) L0 = max(L0, 1u);
        collect_own<VEC>(row, g, sm, leader, rank, C, rank * (CAP / C), CAP / C, L0, NO_LIMIT, keyf, true, true,
                         warp, lane, tid);
        cluster_sync();  // every region and count is in every CTA
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
        } else if (tp < 1.f) {
            // Top-p: the largest t with mass(key >= t) >= top_p * M; top_p <= 0 keeps the
            // maximum alone (the smallest positive target).
            Search st = search_start(maxkey, M, V);
            const float target = tp > 0.f ? tp * M : __uint_as_float(1u);
            threshold_search<VEC, false, true, true>(row, g, sm, C, st, 0, target, keyf, warp, lane, tid);
            t = uint32_t(st.lo);
            denom = st.mass_lo;
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
    fs_status st = make_plan(batch, vocab, fn, KIND != K_TOPP, p);
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
