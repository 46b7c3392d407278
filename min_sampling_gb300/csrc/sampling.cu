// Dual-pivot rejection sampler (sm_103a).
//
// One thread-block cluster per output row; see fs_device.cuh for the layout.
// Steps, in the order the pages give them:
//   pass 1   every CTA reads its share of the row once: per-segment maximum key and
//            mass, the row total M, the positive count and a NaN/negative flag;
//   prologue (top-k-first only) the exact k-th largest value t_k and
//            F_k = mass(x >= t_k) ([explainer] filter order).  Each CTA bounds t_k
//            from below by the k-th largest of its own segment maxima (any subset's
//            k-th largest is at most the row's), keeps its elements at or above that
//            bound, and rank 0 gathers the survivors of the best bound and counts t_k
//            exactly among them;
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
    int shift;                // log2(blocks per segment)
    int ns;                   // segments per row
    int nsc;                  // segments per CTA
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

// Rank 0 takes over the lists of all ranks (u[cnt_idx] of the last exchange holds
// their lengths), keeping keys >= keep; then the cluster barrier after which the
// other CTAs may leave.  Returns the list length on rank 0.
__device__ __forceinline__ int handoff_to_rank0(const Smem& sm, int C, int rank, int cnt_idx, uint32_t keep,
                                                int warp, int lane, int tid) {
    int n = 0;
    if (rank == 0) n = gather_lists(sm, C, cnt_idx, keep, KeyProb(), warp, lane, tid);
    cluster_sync();  // the peers' lists have been read
    return n;
}

// One compact round on rank 0's list (warp-collective): draw, reduce, decide.
// Returns 1 if accepted (token in *j), 0 to continue, -1 if the list had no token
// above low (cannot happen while S_low > 0).
__device__ __forceinline__ int compact_round(const Smem& sm, int n_list, const Pred& f, bool any_filter, float u,
                                             float& low, float& high, float& S_low, int lane, int* j) {
    const int e = locate_in_list(sm.lv, n_list, low, u * S_low, lane);
    if (e < 0) return -1;
    *j = sm.li[e];
    const float pivot1 = sm.lv[e];
    if (!any_filter) return 1;
    const float pivot2 = (pivot1 + high) * 0.5f;
    float M1 = 0.f, M2 = 0.f;
    int C1 = 0, C2 = 0;
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

template <bool VEC>
__global__ void __launch_bounds__(NT, 4) sample_kernel(const SampleArgs a) {
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout L(a.nsc);
    const Smem sm(L);
    const Geom g(a.V, a.shift, a.ns, a.nsc, rank);
    const int V = a.V;
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
    const bool kfirst = a.order == 0 && f.k_on;

    // ---- a2: pass 1, the only HBM read of the row
    int pos = 0;
    bool bad = false;
    if (row_ok) pass1<VEC, true, true>(row, g, sm.segkey, sm.mass[0], warp, lane, pos, bad);
    pos = warp_sum_i(pos);
    const int wbad = __any_sync(FULL, bad) ? 1 : 0;
    if (lane == 0) {
        sm.redi[warp] = pos;
        sm.redi[NW + warp] = wbad;
    }
    __syncthreads();

    // ---- a3 (part 1): local lower bound of t_k and the local candidates
    uint32_t L0c = 0;
    int nloc = -1;  // -1: no candidate list from this CTA
    if (row_ok && kfirst && g.nsc >= k) {
        L0c = max(1u, kth_in_array(sm.segkey, g.nsc, k, sm, warp, lane, tid));
        nloc = compact_ge<VEC, true>(row, g, L0c, keyf, 0.f, sm, warp, lane, tid);
        if (nloc > CAP) nloc = -1;
    }
    if (warp == 0) {
        const int nown = row_ok ? g.nsc : 0;
        const uint32_t km = ordered_max_u(sm.segkey, nown, lane);
        const float s = ordered_sum(sm.mass[0], nown, lane);
        if (lane == 0) {
            int np = 0, nb = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                np += sm.redi[w];
                nb |= sm.redi[NW + w];
            }
            sm.slot[0].f[0] = s;
            sm.slot[0].u[0] = km;
            sm.slot[0].u[1] = uint32_t(nb);
            sm.slot[0].u[2] = uint32_t(np);
            sm.slot[0].u[3] = L0c;
            sm.slot[0].u[4] = uint32_t(nloc);
        }
    }
    int buf = 0;
    exchange(sm, buf, C, tid, 13);
    buf ^= 1;
    uint32_t maxkey = 0, L0 = 0;
    float M = 0.f;
    int npos = 0, ncand = 0;
    bool any_bad = false, lists_ok = true;
    float* cm = reinterpret_cast<float*>(sm.misc + 16);  // per-CTA mass above `low`, rank order
    if (tid < C) cm[tid] = sm.gath[tid].f[0];
    for (int c = 0; c < C; ++c) {
        const Slot& s = sm.gath[c];
        M += s.f[0];
        maxkey = max(maxkey, s.u[0]);
        any_bad |= s.u[1] != 0;
        npos += int(s.u[2]);
        L0 = max(L0, s.u[3]);
        const int n = int(s.u[4]);
        lists_ok = lists_ok && n >= 0;
        ncand += max(n, 0);
    }
    lists_ok = lists_ok && ncand <= CAP;
    __syncthreads();
    const float rowmax = __uint_as_float(maxkey);
    bool valid = row_ok && par_ok && !any_bad && M > 0.f && M <= 3.402823466e38f;
    if (f.m_on) {
        f.t32 = __double2float_ru(double(mp) * double(rowmax));
        if (!(rowmax >= f.t32)) valid = false;  // S is empty: f(max) = 0
    }

    int token = -1, rounds = 0;
    bool accepted = false;
    bool cluster_live = true;  // all CTAs of the cluster still run in lock-step

    if (valid) {
        float low = 0.f, high = rowmax, S_low = M;
        int cur = 0;            // mass[cur][ls] = mass of segment ls above `low`
        int count_low = npos;   // tokens above `low`
        int n_list = 0;
        bool compact = false;
        f.pthr = tp * M;

        // ---- a3 (part 2): exact t_k and F_k
        if (kfirst) {
            if (lists_ok) {
                const int n = handoff_to_rank0(sm, C, rank, 4, L0, warp, lane, tid);
                if (rank != 0) return;
                cluster_live = false;
                compact = true;
                // The list holds every element >= L0, hence every element >= t_k.
                const uint32_t tk = kth_key_in_list(sm, n, k, keyf, warp, lane, tid);
                if (warp == 0) {
                    n_list = filter_list_warp(sm, n, tk, keyf, lane);
                    S_low = ordered_sum(sm.lv, n_list, lane);
                }
                low = 0.f;
            } else {
                // Too many candidates: exact t_k by bit-pattern bisection over the row.
                Bisect st;
                st.lo = L0;  // count(key >= L0) >= k when L0 > 0; count(key >= 0) = V otherwise
                st.hi = uint64_t(maxkey) + 1;
                st.cnt_lo = 0;
                st.mass_lo = 0.f;
                bisect_run<VEC, true, false>(row, g, &st, k, 0.f, keyf, 0.f, sm, &buf, C, warp, lane, tid);
                const uint32_t tk = uint32_t(st.lo);
                mass_count_ge<VEC, true>(row, g, tk, keyf, sm.mass[0], sm, &buf, C, warp, lane, tid, &S_low,
                                         &count_low, cm);
                cur = 0;
                low = tk >= 1u ? __uint_as_float(tk - 1u) : 0.f;  // x > low  <=>  key(x) >= t_k
            }
            f.pthr = tp * S_low;  // top-p inside the k, measured against F_k
        }

        // ---- a4..a7: rejection rounds
        for (int round = 0; round < R_MAX; ++round) {
            if (!compact && count_low <= CAP) {
                // Few tokens left above `low`: gather them (index order) into rank 0.
                const uint32_t thr = prob_key(low) + 1u;
                const int nl = compact_ge<VEC, true>(row, g, thr, keyf, 0.f, sm, warp, lane, tid);
                if (tid == 0) sm.slot[buf].u[0] = uint32_t(min(nl, CAP));
                exchange(sm, buf, C, tid, 9);
                buf ^= 1;
                const int n = handoff_to_rank0(sm, C, rank, 0, thr, warp, lane, tid);
                if (rank != 0) return;
                cluster_live = false;
                compact = true;
                n_list = n;
            }
            const float u = sampler_uniform(a.seed, a.offset, uint32_t(b), uint32_t(round));
            if (compact) {
                // ---- compact rounds: warp 0 of rank 0 on the list
                if (warp != 0) break;
                int j = -1;
                const int st = compact_round(sm, n_list, f, any_filter, u, low, high, S_low, lane, &j);
                if (st < 0) break;
                if (st > 0) {
                    accepted = true;
                    token = j;
                    rounds = round + 1;
                    break;
                }
                continue;
            }

            // ---- a5: draw.  Owner CTA of the target, then segment, then element.
            const float target = u * S_low;
            float acc = 0.f, before = 0.f, lastb = 0.f;
            int owner = -1, lastc = -1;
            for (int c = 0; c < C; ++c) {
                const float m = cm[c];
                if (m > 0.f) {
                    if (owner < 0 && acc + m > target) {
                        owner = c;
                        before = acc;
                    }
                    lastc = c;
                    lastb = acc;
                }
                acc += m;
            }
            bool force = false;
            if (owner < 0) {
                owner = lastc;
                before = lastb;
                force = true;
            }
            if (owner < 0) break;  // no mass above `low` (cannot happen); uniform
            if (rank == owner && warp == 0) {
                const float inf = __int_as_float(0x7f800000);
                const float t = force ? inf : target - before;
                float bseg;
                bool fl;
                const int ls = locate_segment(sm.mass[cur], g.nsc, t, lane, &bseg, &fl);
                const float t2 = (force || fl) ? inf : t - bseg;
                int jj = -1;
                float xx = 0.f;
                if (ls >= 0) locate_in_segment<VEC, true>(row, g, ls, low, t2, lane, &jj, &xx);
                if (lane == 0) {
                    sm.slot[buf].f[0] = xx;
                    sm.slot[buf].u[0] = uint32_t(jj);
                }
            }
            exchange(sm, buf, C, tid, 9);
            buf ^= 1;
            const int j = int(sm.gath[owner].u[0]);
            const float pivot1 = sm.gath[owner].f[0];
            if (j < 0) break;  // uniform: every CTA read the same record
            if (!any_filter) {
                accepted = true;
                token = j;
                rounds = round + 1;
                break;
            }
            const float pivot2 = (pivot1 + high) * 0.5f;

            // ---- a6: fused (mass, count) above pivot1 and pivot2
            const int ia = cur == 0 ? 1 : 0;
            const int ib = cur == 2 ? 1 : 2;
            int c1 = 0, c2 = 0;
            pivot_pass<VEC, true>(row, g, sm.segkey, pivot1, pivot2, sm.mass[ia], sm.mass[ib], warp, lane, c1, c2);
            c1 = warp_sum_i(c1);
            c2 = warp_sum_i(c2);
            if (lane == 0) {
                sm.redi[warp] = c1;
                sm.redi[NW + warp] = c2;
            }
            __syncthreads();
            if (warp == 0) {
                const float t1 = ordered_sum(sm.mass[ia], g.nsc, lane);
                const float t2 = ordered_sum(sm.mass[ib], g.nsc, lane);
                if (lane == 0) {
                    int n1 = 0, n2 = 0;
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        n1 += sm.redi[w];
                        n2 += sm.redi[NW + w];
                    }
                    sm.slot[buf].f[0] = t1;
                    sm.slot[buf].f[1] = t2;
                    sm.slot[buf].u[0] = uint32_t(n1);
                    sm.slot[buf].u[1] = uint32_t(n2);
                }
            }
            exchange(sm, buf, C, tid, 10);
            buf ^= 1;
            float M1 = 0.f, M2 = 0.f;
            int C1 = 0, C2 = 0;
            for (int c = 0; c < C; ++c) {
                M1 += sm.gath[c].f[0];
                M2 += sm.gath[c].f[1];
                C1 += int(sm.gath[c].u[0]);
                C2 += int(sm.gath[c].u[1]);
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
                cur = ia;
                if (tid < C) cm[tid] = sm.gath[tid].f[0];
            } else {
                low = pivot2;
                S_low = M2;
                count_low = C2;
                cur = ib;
                if (tid < C) cm[tid] = sm.gath[tid].f[1];
            }
            __syncthreads();  // cm is read and gath rewritten next round
        }
        if (!accepted) rounds = R_MAX;
    }

    // ---- a8: outputs
    if (cluster_live) cluster_sync();  // no CTA leaves while a peer may read its shared memory
    if (rank == 0 && tid == 0) {
        a.out_token[b] = accepted ? token : -1;
        a.out_valid[b] = accepted ? 1 : 0;
        if (a.out_rounds) a.out_rounds[b] = rounds;
    }
}

// ------------------------------------------------------------------ host side

static fs_status launch_sample(const float* probs, int32_t batch_in, int32_t vocab, const int32_t* indices,
                               int32_t batch_out, const int32_t* top_k, const float* top_p, const float* min_p,
                               int32_t order, uint64_t seed, uint64_t offset, int32_t* out_token, uint8_t* out_valid,
                               int32_t* out_rounds, void* stream) {
    if (batch_out < 0 || batch_in < 0) return FS_ERR_INVALID_ARG;
    if (batch_out == 0) return FS_OK;
    if (!probs || !out_token || !out_valid) return FS_ERR_INVALID_ARG;
    if (vocab < 1) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    if (!indices && batch_out != batch_in) return FS_ERR_INVALID_ARG;
    if (order != FS_ORDER_TOP_K_FIRST && order != FS_ORDER_JOINT) return FS_ERR_INVALID_ARG;

    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(probs) & 15) == 0);
    const void* fn = vec ? reinterpret_cast<const void*>(sample_kernel<true>)
                         : reinterpret_cast<const void*>(sample_kernel<false>);
    Plan p;
    fs_status st = make_plan(batch_out, vocab, fn, p);
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
    a.shift = p.shift;
    a.ns = p.ns;
    a.nsc = p.nsc;
    if (vec) return launch_cluster(sample_kernel<true>, p, batch_out, stream, a);
    return launch_cluster(sample_kernel<false>, p, batch_out, stream, a);
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

}  // extern "C"
