// Filter-only kernels (sm_103a): top_k_renorm_probs, top_p_renorm_probs,
// top_k_mask_logits.
//
// Each finds the exact threshold t on the integer order key of the row's values
// ([drill] sections 2-4: the largest t with count(key >= t) >= k, or with
// mass(key >= t) >= top_p * M), then writes the row once.  One cluster per row:
//   pass 1   one HBM read: per-segment maximum key, the row total and a bad flag;
//   search   top-k: every CTA bounds t from below by the k-th largest of its own
//            segment maxima and keeps its elements at or above that bound; rank 0
//            gathers the survivors of the best bound and counts t exactly among them;
//            a bisection on the key takes over when they do not fit on chip.
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

template <bool VEC, int KIND>
__global__ void __launch_bounds__(NT, 4) filter_kernel(const FilterArgs a) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyLogit, KeyProb>::type;
    constexpr bool IS_PROB = KIND != K_MASK;
    const KEYF keyf;
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout L(a.nsc);
    const Smem sm(L);
    const Geom g(a.V, a.shift, a.ns, a.nsc, rank);
    const int V = a.V;
    const float* row = a.in + size_t(b) * size_t(V);
    float* orow = a.out + size_t(b) * size_t(V);
    const float fill = IS_PROB ? 0.f : __int_as_float(0xff800000);
    const int k = (KIND != K_TOPP) ? a.top_k[b] : 0;
    const float tp = (KIND == K_TOPP) ? a.top_p[b] : 1.f;
    const bool k_on = KIND != K_TOPP && k > 0 && k < V;

    // ---- pass 1
    int pos = 0;
    bool bad = false;
    pass1<VEC, false, IS_PROB>(row, g, sm.segkey, sm.mass[0], warp, lane, pos, bad);
    const int wbad = __any_sync(FULL, bad) ? 1 : 0;
    if (lane == 0) sm.redi[NW + warp] = wbad;
    __syncthreads();

    // Local lower bound of the top-k threshold and the local candidates.
    uint32_t L0c = 0;
    int nloc = -1;
    if (k_on && g.nsc >= k) {
        L0c = max(IS_PROB ? 1u : 0u, kth_in_array(sm.segkey, g.nsc, k, sm, warp, lane, tid));
        nloc = compact_ge<VEC, false>(row, g, L0c, keyf, fill, sm, warp, lane, tid);
        if (nloc > CAP) nloc = -1;
    }
    if (warp == 0) {
        const uint32_t km = ordered_max_u(sm.segkey, g.nsc, lane);
        const float s = IS_PROB ? ordered_sum(sm.mass[0], g.nsc, lane) : 0.f;
        if (lane == 0) {
            int nb = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) nb |= sm.redi[NW + w];
            sm.slot[0].f[0] = s;
            sm.slot[0].u[0] = km;
            sm.slot[0].u[1] = uint32_t(nb);
            sm.slot[0].u[3] = L0c;
            sm.slot[0].u[4] = uint32_t(nloc);
        }
    }
    int buf = 0;
    exchange(sm, buf, C, tid, 13);
    buf ^= 1;
    uint32_t maxkey = 0, L0 = 0;
    float M = 0.f;
    bool any_bad = false, lists_ok = true;
    int ncand = 0;
    for (int c = 0; c < C; ++c) {
        const Slot& s = sm.gath[c];
        M += s.f[0];
        maxkey = max(maxkey, s.u[0]);
        any_bad |= s.u[1] != 0;
        L0 = max(L0, s.u[3]);
        const int n = int(s.u[4]);
        lists_ok = lists_ok && n >= 0;
        ncand += max(n, 0);
    }
    lists_ok = lists_ok && ncand <= CAP;
    __syncthreads();

    bool valid = !any_bad;
    if (IS_PROB) valid = valid && M > 0.f && M <= 3.402823466e38f;
    if (KIND == K_TOPP && isnan(tp)) valid = false;

    uint32_t t = 0;   // keep key >= t
    float denom = M;  // kept mass (probabilities)
    if (valid) {
        if (KIND != K_TOPP) {
            if (k_on) {
                if (lists_ok) {
                    if (rank == 0) {
                        const int n = gather_lists(sm, C, 4, L0, keyf, warp, lane, tid);
                        const uint32_t tk = kth_key_in_list(sm, n, k, keyf, warp, lane, tid);
                        if (warp == 0) {
                            float s = 0.f;
                            for (int i = lane; i < n; i += 32) s += keyf(sm.lv[i]) >= tk ? sm.lv[i] : 0.f;
                            s = warp_sum(s);
                            if (lane == 0) {
                                sm.slot[buf].f[0] = s;
                                sm.slot[buf].u[0] = tk;
                            }
                        }
                    }
                    exchange(sm, buf, C, tid, 9);
                    buf ^= 1;
                    t = sm.gath[0].u[0];
                    denom = sm.gath[0].f[0];
                    __syncthreads();
                } else {
                    Bisect st;
                    st.lo = L0;  // crit(L0) holds (L0 <= t_k), and crit(0) trivially
                    st.hi = uint64_t(maxkey) + 1;
                    st.cnt_lo = 0;
                    st.mass_lo = 0.f;
                    bisect_run<VEC, false, false>(row, g, &st, k, 0.f, keyf, fill, sm, &buf, C, warp, lane, tid);
                    t = uint32_t(st.lo);
                    if (IS_PROB) {
                        int cnt;
                        mass_count_ge<VEC, false>(row, g, t, keyf, nullptr, sm, &buf, C, warp, lane, tid, &denom,
                                                  &cnt, nullptr);
                    }
                }
            }
        } else {
            if (tp >= 1.f) {
                t = 0;
                denom = M;
            } else if (tp <= 0.f) {
                t = maxkey;
                int cnt;
                mass_count_ge<VEC, false>(row, g, t, keyf, nullptr, sm, &buf, C, warp, lane, tid, &denom, &cnt,
                                          nullptr);
            } else {
                Bisect st;
                st.lo = 0;
                st.hi = uint64_t(maxkey) + 1;
                st.cnt_lo = 0;
                st.mass_lo = M;
                bisect_run<VEC, false, true>(row, g, &st, 0, tp * M, keyf, 0.f, sm, &buf, C, warp, lane, tid);
                t = uint32_t(st.lo);
                denom = st.mass_lo;
            }
        }
    }

    // ---- write this CTA's share of the row
    const bool vec_out = VEC && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
    visit<TRIP, VEC, false>(
        row, g, fill, warp, lane, [&](int ls) { return valid && sm.segkey[ls] >= t; },
        [&](int, int, int base, float4 x, bool on) {
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xv = q_at(x, q);
                o[q] = (on && keyf(xv) >= t) ? (IS_PROB ? xv / denom : xv) : fill;
            }
            if (vec_out && base + 3 < V) {
                *reinterpret_cast<float4*>(orow + base) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (base + q < V) orow[base + q] = o[q];
            }
        },
        [](int, bool) {});
    if (rank == 0 && tid == 0 && a.out_valid) a.out_valid[b] = valid ? 1 : 0;
    cluster_sync();  // no CTA leaves while a peer may read its shared memory
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
    fs_status st = make_plan(batch, vocab, fn, p);
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
