// Filter-only kernels (sm_103a): top_k_renorm_probs, top_p_renorm_probs,
// top_k_mask_logits.
//
// Each finds the exact threshold t on the integer order key of the row's values
// ([drill] sections 2-4: the largest t with count(key >= t) >= k, or with
// mass(key >= t) >= top_p * M), then writes the row once.  One cluster per row:
//   pass 1   one HBM read: per-segment maximum key, the row total and a bad flag;
//   search   top-k: candidates = every element at or above the k-th largest segment
//            maximum (a lower bound of t), gathered into rank 0, where t is exact by
//            counting; a bisection on the key takes over if they do not fit.
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
    int nsc;
    int ns;
};

struct KeyP {
    __device__ __forceinline__ uint32_t operator()(float x) const { return prob_key(x); }
};
struct KeyL {
    __device__ __forceinline__ uint32_t operator()(float x) const { return logit_key(x); }
};

// Mass (probabilities) and count of key >= t over this CTA's segments, cluster-wide.
template <bool VEC, typename KEYF>
__device__ void mass_count_ge(const float* __restrict__ row, int V, int s0, int nsc, const uint32_t* segkey,
                              uint32_t t, KEYF keyf, const Smem& sm, int& buf, int C, int warp, int lane,
                              int tid, float& mass, int& cnt) {
    float wm = 0.f;
    int wc = 0;
    for (int ls = warp; ls < nsc; ls += NW) {
        if (segkey[ls] < t) continue;
        float v[SEG_IT][4];
        load_segment<VEC, false>(row, V, s0 + ls, lane, 0.f, v);
        float m = 0.f;
        int c = 0;
        const int base0 = (s0 + ls) * SEG + lane * 4;
#pragma unroll
        for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool g = keyf(v[it][q]) >= t && base0 + it * 128 + q < V;
                m += g ? v[it][q] : 0.f;
                c += g;
            }
        wm += warp_sum(m);
        wc += warp_sum_i(c);
    }
    if (lane == 0) {
        sm.redf[warp] = wm;
        sm.redi[warp] = wc;
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        int n = 0;
        for (int w = 0; w < NW; ++w) { s += sm.redf[w]; n += sm.redi[w]; }
        sm.slot[buf].f[0] = s;
        sm.slot[buf].u[0] = uint32_t(n);
    }
    exchange(sm, buf, C, warp, lane);
    buf ^= 1;
    mass = 0.f;
    cnt = 0;
    for (int c = 0; c < C; ++c) {
        mass += sm.gath[c].f[0];
        cnt += int(sm.gath[c].u[0]);
    }
    __syncthreads();
}

template <bool VEC, int KIND>
__global__ void __launch_bounds__(NT, 1) filter_kernel(const FilterArgs a) {
    using KEYF = typename std::conditional<KIND == K_MASK, KeyL, KeyP>::type;
    const KEYF keyf;
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout L(a.nsc, a.ns);
    const Smem sm(L);
    const int V = a.V, NS = a.ns;
    const int s0 = rank * a.nsc;
    const int nsc = max(0, min(a.nsc, NS - s0));
    const float* row = a.in + size_t(b) * size_t(V);
    float* orow = a.out + size_t(b) * size_t(V);
    const bool is_prob = KIND != K_MASK;

    // ---- pass 1
    if (tid == 0) sm.misc[1] = 0;
    __syncthreads();
    for (int ls = warp; ls < nsc; ls += NW) {
        float v[SEG_IT][4];
        load_segment<VEC, false>(row, V, s0 + ls, lane, is_prob ? 0.f : __int_as_float(0xff800000), v);
        uint32_t kmax = 0;
        float s = 0.f;
        bool bad = false;
        const int base0 = (s0 + ls) * SEG + lane * 4;
#pragma unroll
        for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = v[it][q];
                const bool inr = base0 + it * 128 + q < V;
                if (is_prob) {
                    bad |= !(x >= 0.f);
                    s += x;
                } else {
                    bad |= isnan(x);
                }
                kmax = max(kmax, inr ? keyf(x) : 0u);
            }
        kmax = warp_max_u(kmax);
        if (is_prob) s = warp_sum(s);
        if (__any_sync(FULL, bad) && lane == 0) sm.misc[1] = 1;
        if (lane == 0) {
            sm.segkey[ls] = kmax;
            sm.mass[0][ls] = s;
        }
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t km = 0;
        for (int base = 0; base < nsc; base += 32) km = max(km, base + lane < nsc ? sm.segkey[base + lane] : 0u);
        km = warp_max_u(km);
        const float s = ordered_sum(sm.mass[0], nsc, lane);
        if (lane == 0) {
            sm.slot[0].u[0] = km;
            sm.slot[0].f[1] = s;
            sm.slot[0].u[1] = uint32_t(sm.misc[1]);
        }
    }
    int buf = 0;
    exchange(sm, buf, C, warp, lane);
    buf ^= 1;
    uint32_t maxkey = 0;
    float M = 0.f;
    bool bad = false;
    for (int c = 0; c < C; ++c) {
        maxkey = max(maxkey, sm.gath[c].u[0]);
        M += sm.gath[c].f[1];
        bad |= sm.gath[c].u[1] != 0;
    }
    __syncthreads();

    bool valid = !bad;
    if (is_prob) valid = valid && M > 0.f && M <= 3.402823466e38f;
    const int k = (KIND != K_TOPP && a.top_k) ? a.top_k[b] : 0;
    const float tp = (KIND == K_TOPP && a.top_p) ? a.top_p[b] : 1.f;
    if (KIND == K_TOPP && isnan(tp)) valid = false;

    uint32_t t = 0;       // keep key >= t
    float denom = M;      // kept mass (probabilities)
    if (valid) {
        if (KIND != K_TOPP) {
            if (k > 0 && k < V) {
                // Candidates: everything at or above the k-th largest segment maximum.
                uint32_t L0 = is_prob ? 1u : 0u;
                const bool pruned = k <= NS;
                if (pruned) {
                    gather_segkeys(sm, a.nsc, NS, tid);
                    L0 = max(L0, kth_key_in_array(sm.segall, NS, k, sm, warp, lane, tid));
                }
                const int nloc = compact_ge<VEC, false>(row, V, s0, nsc, sm.segkey, L0, keyf,
                                                        is_prob ? 0.f : __int_as_float(0xff800000), sm, warp,
                                                        lane, tid);
                if (tid == 0) sm.slot[buf].u[0] = uint32_t(nloc);
                exchange(sm, buf, C, warp, lane);
                buf ^= 1;
                int ntot = 0;
                for (int c = 0; c < C; ++c) ntot += int(sm.gath[c].u[0]);
                __syncthreads();
                if (ntot <= CAP) {
                    if (rank == 0) {
                        gather_lists(sm, C, tid);
                        uint32_t tk = kth_key_in_list(sm, ntot, k, keyf, warp, lane, tid);
                        if (warp == 0) {
                            float s = 0.f;
                            for (int base = 0; base < ntot; base += 32) {
                                const int i = base + lane;
                                const bool g = i < ntot && keyf(sm.lv[i]) >= tk;
                                s += warp_sum(g ? sm.lv[i] : 0.f);
                            }
                            if (lane == 0) {
                                sm.slot[buf].u[0] = tk;
                                sm.slot[buf].f[0] = s;
                            }
                        }
                    }
                    exchange(sm, buf, C, warp, lane);
                    buf ^= 1;
                    t = sm.gath[0].u[0];
                    denom = sm.gath[0].f[0];
                    __syncthreads();
                } else {
                    Bisect st;
                    st.lo = pruned ? L0 : 0u;
                    st.hi = uint64_t(maxkey) + 1;
                    st.cnt_lo = 0;
                    st.mass_lo = 0.f;
                    bisect_run<VEC, false, false>(row, V, s0, nsc, sm.segkey, st, k, 0.f, keyf,
                                                  is_prob ? 0.f : __int_as_float(0xff800000), sm, buf, C, warp,
                                                  lane, tid);
                    t = uint32_t(st.lo);
                    if (is_prob) {
                        int cnt;
                        mass_count_ge<VEC>(row, V, s0, nsc, sm.segkey, t, keyf, sm, buf, C, warp, lane, tid,
                                           denom, cnt);
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
                mass_count_ge<VEC>(row, V, s0, nsc, sm.segkey, t, keyf, sm, buf, C, warp, lane, tid, denom, cnt);
            } else {
                Bisect st;
                st.lo = 0;
                st.hi = uint64_t(maxkey) + 1;
                st.cnt_lo = 0;
                st.mass_lo = M;
                bisect_run<VEC, false, true>(row, V, s0, nsc, sm.segkey, st, 0, tp * M, keyf, 0.f, sm, buf, C,
                                             warp, lane, tid);
                t = uint32_t(st.lo);
                denom = st.mass_lo;
            }
        }
    }

    // ---- write this CTA's share of the row
    const float fill = is_prob ? 0.f : __int_as_float(0xff800000);
    const bool vec_out = VEC && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
    for (int ls = warp; ls < nsc; ls += NW) {
        const int s = s0 + ls;
        const bool any_kept = valid && sm.segkey[ls] >= t;
        float v[SEG_IT][4];
        if (any_kept) {
            load_segment<VEC, false>(row, V, s, lane, 0.f, v);
        }
#pragma unroll
        for (int it = 0; it < SEG_IT; ++it) {
            const int base = s * SEG + it * 128 + lane * 4;
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (!any_kept) {
                    o[q] = fill;
                } else {
                    const float x = v[it][q];
                    const bool keep = keyf(x) >= t;
                    o[q] = keep ? (is_prob ? x / denom : x) : fill;
                }
            }
            if (vec_out && base + 3 < V) {
                *reinterpret_cast<float4*>(orow + base) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (base + q < V) orow[base + q] = o[q];
            }
        }
    }
    if (rank == 0 && tid == 0 && a.out_valid) a.out_valid[b] = valid ? 1 : 0;
    cluster_sync();   // no CTA leaves while a peer may read its shared memory
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
    Plan p;
    fs_status st = make_plan(batch, vocab, p);
    if (st != FS_OK) return st;
    FilterArgs a;
    a.in = in;
    a.out = out;
    a.V = vocab;
    a.top_k = top_k;
    a.top_p = top_p;
    a.out_valid = out_valid;
    a.nsc = p.nsc;
    a.ns = p.ns;
    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(in) & 15) == 0);
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
