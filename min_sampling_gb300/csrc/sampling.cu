// Dual-pivot rejection sampler (sm_103a).
//
// One thread-block cluster per output row; see fs_device.cuh for the layout.
// Steps, in the order the pages give them:
//   pass 1   every CTA reads its share of the row once: per-segment maximum and
//            mass, the row total M, the positive count and a NaN/negative flag;
//   prologue (top-k-first only) the exact k-th largest value t_k and
//            F_k = mass(x >= t_k) ([explainer] filter order), from a candidate list
//            bounded below by the k-th largest segment maximum;
//   rounds   ([blog] dual-pivot rejection sampling) draw j by inverse transform over
//            {p > low}, pivot1 = p_j, pivot2 = (pivot1 + high) / 2, one fused
//            reduction of (mass, count) above both pivots, then accept j, or
//            (low, high) <- (pivot1, pivot2), or low <- pivot2.
// While many tokens lie above `low` a round visits only segments whose maximum is
// above pivot1 (read again through L2); once at most CAP tokens are left they are
// gathered, in index order, into rank 0's shared memory and the remaining rounds run
// there on one warp, with no further cluster traffic.
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
    int* out_token;
    unsigned char* out_valid;
    int* out_rounds;
    int nsc;                  // segments per CTA
    int ns;                   // segments per row
};

// The acceptance test f(tau) ([blog] rejection sampling: count / remaining mass above
// the pivot; [explainer] Top-k, Top-p, Min-p), from the count and the mass of the
// tokens strictly above tau.
struct Pred {
    bool k_on, p_on, m_on;
    int k;
    float pthr;   // top_p * M'   (M' = M, or F_k for top-k-first)
    float t32;    // min-p threshold: float32 rounded up from min_p * max
    __device__ __forceinline__ bool operator()(int cnt, float mass, float tau) const {
        if (k_on && !(cnt < k)) return false;
        if (p_on && !(cnt == 0 || mass < pthr)) return false;
        if (m_on && !(tau >= t32)) return false;
        return true;
    }
};

struct KeyProb {
    __device__ __forceinline__ uint32_t operator()(float x) const { return prob_key(x); }
};

template <bool VEC>
__global__ void __launch_bounds__(NT, 1) sample_kernel(const SampleArgs a) {
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout L(a.nsc, a.ns);
    const Smem sm(L);
    const int V = a.V, NS = a.ns;
    const int s0 = rank * a.nsc;
    const int nsc = max(0, min(a.nsc, NS - s0));
    const KeyProb keyf;

    // ---- a1: row map and per-row parameters
    const int r = a.indices ? a.indices[b] : b;
    const bool row_ok = r >= 0 && r < a.batch_in;
    const float* row = a.probs + size_t(row_ok ? r : 0) * size_t(V);
    const int k = a.top_k ? a.top_k[b] : 0;
    const float tp = a.top_p ? a.top_p[b] : 1.f;
    const float mp = a.min_p ? a.min_p[b] : 0.f;
    Pred f;
    f.k_on = k > 0 && k < V;
    f.k = k;
    f.p_on = tp < 1.f;
    f.m_on = mp > 0.f;
    f.pthr = 0.f;
    f.t32 = 0.f;
    const bool par_ok = !isnan(tp) && !isnan(mp);
    const bool any_filter = f.k_on || f.p_on || f.m_on;

    // ---- a2: pass 1 (the only HBM read of the row)
    if (tid == 0) sm.misc[1] = 0;
    __syncthreads();
    int wpos = 0;
    if (row_ok) {
        for (int ls = warp; ls < nsc; ls += NW) {
            float v[SEG_IT][4];
            load_segment<VEC, true>(row, V, s0 + ls, lane, 0.f, v);
            uint32_t kmax = 0;
            float s = 0.f;
            int pos = 0;
            bool bad = false;
#pragma unroll
            for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x = v[it][q];
                    bad |= !(x >= 0.f);
                    kmax = max(kmax, prob_key(x));
                    s += x;
                    pos += x > 0.f;
                }
            kmax = warp_max_u(kmax);
            s = warp_sum(s);
            wpos += warp_sum_i(pos);
            if (__any_sync(FULL, bad) && lane == 0) sm.misc[1] = 1;
            if (lane == 0) {
                sm.segkey[ls] = kmax;
                sm.mass[0][ls] = s;
            }
        }
    }
    if (lane == 0) sm.redi[warp] = wpos;
    __syncthreads();
    if (warp == 0) {
        uint32_t km = 0;
        for (int base = 0; base < nsc; base += 32) km = max(km, base + lane < nsc ? sm.segkey[base + lane] : 0u);
        km = warp_max_u(km);
        const float s = ordered_sum(sm.mass[0], nsc, lane);
        if (lane == 0) {
            int np = 0;
            for (int w = 0; w < NW; ++w) np += sm.redi[w];
            sm.slot[0].u[0] = km;
            sm.slot[0].f[1] = s;
            sm.slot[0].u[1] = uint32_t(sm.misc[1]);
            sm.slot[0].u[2] = uint32_t(np);
        }
    }
    int buf = 0;
    exchange(sm, buf, C, warp, lane);
    buf ^= 1;
    uint32_t maxkey = 0;
    float M = 0.f;
    bool bad = false;
    int npos = 0;
    float cm[MAX_CLUSTER];
#pragma unroll
    for (int c = 0; c < MAX_CLUSTER; ++c) {
        cm[c] = 0.f;
        if (c < C) {
            maxkey = max(maxkey, sm.gath[c].u[0]);
            M += sm.gath[c].f[1];
            bad |= sm.gath[c].u[1] != 0;
            npos += int(sm.gath[c].u[2]);
            cm[c] = sm.gath[c].f[1];
        }
    }
    const float rowmax = __uint_as_float(maxkey);
    bool valid = row_ok && par_ok && !bad && M > 0.f && M <= 3.402823466e38f;
    if (f.m_on) {
        f.t32 = __double2float_ru(double(mp) * double(rowmax));
        if (!(rowmax >= f.t32)) valid = false;     // S is empty: f(max) = 0
    }

    int token = -1, rounds = 0;
    bool accepted = false;
    bool cluster_live = true;   // all CTAs of the cluster still run in lock-step

    if (valid) {
        float low = 0.f, high = rowmax, S_low = M;
        int cur = 0;            // mass[cur][ls] = mass of segment ls above `low`
        int count_low = npos;   // tokens above `low`
        int n_list = 0;
        bool compact = false;
        f.pthr = tp * M;

        // ---- a3: top-k-first prologue
        if (a.order == 0 && f.k_on) {
            uint32_t L0 = 1u;   // default: every positive element is a candidate
            const bool pruned = k <= NS;
            if (pruned) {
                gather_segkeys(sm, a.nsc, NS, tid);
                L0 = max(1u, kth_key_in_array(sm.segall, NS, k, sm, warp, lane, tid));
            }
            const int nloc = compact_ge<VEC, true>(row, V, s0, nsc, sm.segkey, L0, keyf, 0.f, sm, warp, lane, tid);
            if (tid == 0) sm.slot[buf].u[0] = uint32_t(nloc);
            exchange(sm, buf, C, warp, lane);
            buf ^= 1;
            int ntot = 0;
            for (int c = 0; c < C; ++c) ntot += int(sm.gath[c].u[0]);
            if (ntot <= CAP) {
                if (rank == 0) gather_lists(sm, C, tid);
                cluster_sync();            // peers' lists are read; they may leave now
                if (rank != 0) return;
                cluster_live = false;
                compact = true;
                // Exact t_k on the candidates (they hold every element >= t_k).
                const uint32_t tk = kth_key_in_list(sm, ntot, k, keyf, warp, lane, tid);
                if (warp == 0) {
                    int w = 0;
                    for (int base = 0; base < ntot; base += 32) {
                        const int i = base + lane;
                        const bool keep = i < ntot && keyf(sm.lv[i]) >= tk;
                        const float xv = keep ? sm.lv[i] : 0.f;
                        const int xi = keep ? sm.li[i] : 0;
                        const unsigned bal = __ballot_sync(FULL, keep);
                        const int pos = w + __popc(bal & ((1u << lane) - 1u));
                        __syncwarp();
                        if (keep) { sm.lv[pos] = xv; sm.li[pos] = xi; }
                        __syncwarp();
                        w += __popc(bal);
                    }
                    n_list = w;
                    S_low = ordered_sum(sm.lv, n_list, lane);
                }
                low = 0.f;
            } else {
                // Too many candidates: exact t_k by bit-pattern bisection over the row.
                Bisect st;
                st.lo = pruned ? L0 : 0u;
                st.hi = uint64_t(maxkey) + 1;
                st.cnt_lo = 0;
                st.mass_lo = 0.f;
                bisect_run<VEC, true, false>(row, V, s0, nsc, sm.segkey, st, k, 0.f, keyf, 0.f, sm, buf, C,
                                             warp, lane, tid);
                const uint32_t tk = uint32_t(st.lo);
                // Per-segment mass of {key >= t_k}; F_k and the count.
                int wc = 0;
                for (int ls = warp; ls < nsc; ls += NW) {
                    float m = 0.f;
                    int c = 0;
                    if (sm.segkey[ls] >= tk) {
                        float v[SEG_IT][4];
                        load_segment<VEC, true>(row, V, s0 + ls, lane, 0.f, v);
#pragma unroll
                        for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const bool g = keyf(v[it][q]) >= tk && v[it][q] > 0.f;
                                m += g ? v[it][q] : 0.f;
                                c += g;
                            }
                        m = warp_sum(m);
                        c = warp_sum_i(c);
                    }
                    if (lane == 0) sm.mass[0][ls] = m;
                    wc += c;
                }
                if (lane == 0) sm.redi[warp] = wc;
                __syncthreads();
                if (warp == 0) {
                    const float s = ordered_sum(sm.mass[0], nsc, lane);
                    if (lane == 0) {
                        int n = 0;
                        for (int w = 0; w < NW; ++w) n += sm.redi[w];
                        sm.slot[buf].f[0] = s;
                        sm.slot[buf].u[0] = uint32_t(n);
                    }
                }
                exchange(sm, buf, C, warp, lane);
                buf ^= 1;
                S_low = 0.f;
                count_low = 0;
#pragma unroll
                for (int c = 0; c < MAX_CLUSTER; ++c) {
                    cm[c] = c < C ? sm.gath[c].f[0] : 0.f;
                    if (c < C) {
                        S_low += sm.gath[c].f[0];
                        count_low += int(sm.gath[c].u[0]);
                    }
                }
                cur = 0;
                low = tk >= 1u ? __uint_as_float(tk - 1u) : 0.f;   // x > low  <=>  key(x) >= t_k
            }
            f.pthr = tp * S_low;   // top-p inside the k, measured against F_k
        }

        // ---- a4..a7: rejection rounds
        for (int round = 0; round < R_MAX; ++round) {
            if (!compact && count_low <= CAP) {
                // Few tokens left above `low`: gather them (index order) into rank 0.
                const uint32_t thr = prob_key(low) + 1u;
                const int nloc = compact_ge<VEC, true>(row, V, s0, nsc, sm.segkey, thr, keyf, 0.f, sm, warp, lane, tid);
                if (tid == 0) sm.slot[buf].u[0] = uint32_t(nloc);
                exchange(sm, buf, C, warp, lane);
                buf ^= 1;
                int ntot = 0;
                for (int c = 0; c < C; ++c) ntot += int(sm.gath[c].u[0]);
                if (rank == 0) gather_lists(sm, C, tid);
                cluster_sync();
                if (rank != 0) return;
                cluster_live = false;
                compact = true;
                n_list = min(ntot, CAP);
            }
            if (compact && warp != 0) break;

            const float u = sampler_uniform(a.seed, a.offset, uint32_t(b), uint32_t(round));
            const float target = u * S_low;
            int j;
            float pivot1;
            if (compact) {
                // ---- compact round: warp 0 of rank 0 on the list
                const int e = locate_in_list(sm.lv, n_list, low, target, lane);
                if (e < 0) break;   // no token above `low` (cannot happen while S_low > 0)
                j = sm.li[e];
                pivot1 = sm.lv[e];
            } else {
                // ---- a5: draw. Owner CTA of the target, then segment, then element.
                float acc = 0.f, before = 0.f, lastb = 0.f;
                int owner = -1, lastc = -1;
#pragma unroll
                for (int c = 0; c < MAX_CLUSTER; ++c) {
                    if (c < C) {
                        const float m = cm[c];
                        if (m > 0.f) {
                            if (owner < 0 && acc + m > target) { owner = c; before = acc; }
                            lastc = c;
                            lastb = acc;
                        }
                        acc += m;
                    }
                }
                bool force = false;
                if (owner < 0) { owner = lastc; before = lastb; force = true; }
                if (owner < 0) break;   // no mass above `low` (cannot happen); uniform
                if (rank == owner && warp == 0) {
                    const float t = force ? __int_as_float(0x7f800000) : target - before;
                    float bseg;
                    bool fl;
                    const int ls = locate_segment(sm.mass[cur], nsc, t, lane, bseg, fl);
                    const float t2 = (force || fl) ? __int_as_float(0x7f800000) : t - bseg;
                    int jj = -1;
                    float xx = 0.f;
                    if (ls >= 0) locate_in_segment<VEC, true>(row, V, s0 + ls, low, t2, lane, jj, xx);
                    if (lane == 0) {
                        sm.slot[buf].u[0] = uint32_t(jj);
                        sm.slot[buf].f[0] = xx;
                    }
                }
                exchange(sm, buf, C, warp, lane);
                buf ^= 1;
                j = int(sm.gath[owner].u[0]);
                pivot1 = sm.gath[owner].f[0];
                if (j < 0) break;   // uniform: every CTA read the same record
            }
            const float pivot2 = (pivot1 + high) * 0.5f;
            if (!any_filter) {
                accepted = true;
                token = j;
                rounds = round + 1;
                break;
            }

            // ---- a6: fused (mass, count) above pivot1 and pivot2
            float M1 = 0.f, M2 = 0.f;
            int C1 = 0, C2 = 0;
            float cm1[MAX_CLUSTER], cm2[MAX_CLUSTER];
            const int ia = cur == 0 ? 1 : 0;
            const int ib = cur == 2 ? 1 : 2;
            if (compact) {
                for (int i = lane; i < n_list; i += 32) {
                    const float x = sm.lv[i];
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
            } else {
                int wc1 = 0, wc2 = 0;
                for (int ls = warp; ls < nsc; ls += NW) {
                    float m1 = 0.f, m2 = 0.f;
                    int c1 = 0, c2 = 0;
                    if (sm.segkey[ls] > prob_key(pivot1)) {
                        float v[SEG_IT][4];
                        load_segment<VEC, true>(row, V, s0 + ls, lane, 0.f, v);
#pragma unroll
                        for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float x = v[it][q];
                                const bool g1 = x > pivot1, g2 = x > pivot2;
                                m1 += g1 ? x : 0.f;
                                m2 += g2 ? x : 0.f;
                                c1 += g1;
                                c2 += g2;
                            }
                        m1 = warp_sum(m1);
                        m2 = warp_sum(m2);
                        c1 = warp_sum_i(c1);
                        c2 = warp_sum_i(c2);
                    }
                    if (lane == 0) {
                        sm.mass[ia][ls] = m1;
                        sm.mass[ib][ls] = m2;
                    }
                    wc1 += c1;
                    wc2 += c2;
                }
                if (lane == 0) {
                    sm.redi[warp * 4 + 0] = wc1;
                    sm.redi[warp * 4 + 1] = wc2;
                }
                __syncthreads();
                if (warp == 0) {
                    const float s1 = ordered_sum(sm.mass[ia], nsc, lane);
                    const float s2 = ordered_sum(sm.mass[ib], nsc, lane);
                    if (lane == 0) {
                        int n1 = 0, n2 = 0;
                        for (int w = 0; w < NW; ++w) { n1 += sm.redi[w * 4 + 0]; n2 += sm.redi[w * 4 + 1]; }
                        sm.slot[buf].f[0] = s1;
                        sm.slot[buf].f[1] = s2;
                        sm.slot[buf].u[0] = uint32_t(n1);
                        sm.slot[buf].u[1] = uint32_t(n2);
                    }
                }
                exchange(sm, buf, C, warp, lane);
                buf ^= 1;
#pragma unroll
                for (int c = 0; c < MAX_CLUSTER; ++c) {
                    cm1[c] = c < C ? sm.gath[c].f[0] : 0.f;
                    cm2[c] = c < C ? sm.gath[c].f[1] : 0.f;
                    if (c < C) {
                        M1 += sm.gath[c].f[0];
                        M2 += sm.gath[c].f[1];
                        C1 += int(sm.gath[c].u[0]);
                        C2 += int(sm.gath[c].u[1]);
                    }
                }
            }

            // ---- a7: the three cases
            if (f(C1, M1, pivot1)) {
                accepted = true;
                token = j;
                rounds = round + 1;
                break;
            }
            if (f(C2, M2, pivot2)) {
                low = pivot1;
                high = pivot2;
                S_low = M1;
                count_low = C1;
                if (!compact) {
                    cur = ia;
#pragma unroll
                    for (int c = 0; c < MAX_CLUSTER; ++c) cm[c] = cm1[c];
                }
            } else {
                low = pivot2;
                S_low = M2;
                count_low = C2;
                if (!compact) {
                    cur = ib;
#pragma unroll
                    for (int c = 0; c < MAX_CLUSTER; ++c) cm[c] = cm2[c];
                }
            }
            if (!compact) __syncthreads();   // gath / mass buffers are rewritten next round
        }
        if (!accepted) rounds = R_MAX;
    }

    // ---- a8: outputs
    if (cluster_live) cluster_sync();   // no CTA leaves while a peer may read its shared memory
    if (rank == 0 && tid == 0) {
        a.out_token[b] = accepted ? token : -1;
        a.out_valid[b] = accepted ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = rounds;
    }
}

// ------------------------------------------------------------------ host side

static fs_status launch_sample(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                               int32_t batch_out, const int32_t* top_k, const float* top_p,
                               const float* min_p, int32_t order, uint64_t seed, uint64_t offset,
                               int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (batch_out < 0 || batch_in < 0) return FS_ERR_INVALID_ARG;
    if (batch_out == 0) return FS_OK;
    if (!probs || !out_token || !out_valid) return FS_ERR_INVALID_ARG;
    if (vocab < 1) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    if (!indices && batch_out != batch_in) return FS_ERR_INVALID_ARG;
    if (order != FS_ORDER_TOP_K_FIRST && order != FS_ORDER_JOINT) return FS_ERR_INVALID_ARG;

    Plan p;
    fs_status st = make_plan(batch_out, vocab, p);
    if (st != FS_OK) return st;
    SampleArgs a;
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
    a.out_token = out_token;
    a.out_valid = out_valid;
    a.out_rounds = out_rounds;
    a.nsc = p.nsc;
    a.ns = p.ns;
    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(probs) & 15) == 0);
    if (vec) return launch_cluster(sample_kernel<true>, p, batch_out, stream, a);
    return launch_cluster(sample_kernel<false>, p, batch_out, stream, a);
}

}  // namespace fsd

extern "C" {

fs_status fs_sampling_from_probs(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                 int32_t batch_out, uint64_t seed, uint64_t offset, int32_t* out_token,
                                 uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, nullptr, nullptr,
                              FS_ORDER_JOINT, seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_k_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const int32_t* top_k, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!top_k && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, nullptr, nullptr,
                              FS_ORDER_JOINT, seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const float* top_p, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!top_p && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, top_p, nullptr,
                              FS_ORDER_JOINT, seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_min_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                            int32_t batch_out, const float* min_p, uint64_t seed, uint64_t offset,
                            int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if (!min_p && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, nullptr, nullptr, min_p,
                              FS_ORDER_JOINT, seed, offset, out_token, out_valid, out_rounds, stream);
}

fs_status fs_top_k_top_p_sampling(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                                  int32_t batch_out, const int32_t* top_k, const float* top_p,
                                  const float* min_p, int32_t order, uint64_t seed, uint64_t offset,
                                  int32_t* out_token, uint8_t* out_valid, int32_t* out_rounds, void* stream) {
    if ((!top_k || !top_p) && batch_out > 0) return FS_ERR_INVALID_ARG;
    return fsd::launch_sample(probs, batch_in, vocab, indices, batch_out, top_k, top_p, min_p, order, seed,
                              offset, out_token, out_valid, out_rounds, stream);
}

}  // extern "C"
