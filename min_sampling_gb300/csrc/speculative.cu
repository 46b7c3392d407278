// Chain speculative-sampling verification (sm_103a).
//
// The pages name speculative-decoding verification as a use of the sorting-free
// sampler ([blog] section on community adoption) without giving its algorithm; this
// kernel follows the published method (Leviathan, Kalman, Matias, "Fast Inference
// from Transformers via Speculative Decoding", ICML 2023, Algorithm 1; Chen et al.,
// "Accelerating Large Language Model Decoding with Speculative Sampling", 2023,
// Algorithm 2).  Per batch row, L draft tokens d_i drawn from draft rows q_i and
// L + 1 target rows p_i:
//   accept d_i while u_i * q_i(d_i) < p_i(d_i) (probability min(1, p/q));
//   at the first rejection i, emit a token drawn from the residual max(p_i - q_i, 0);
//   after L acceptances, emit a token drawn from p_{L+1}.
// The final draw is the sampler's own: one streaming pass over the row of weights
// (the residual is formed at the loads, Geom::qrow), per-segment masses into the
// leader, then the inverse transform over CTAs, segments and tokens (draw_full).
//
// One cluster per batch row.  Every CTA runs the L acceptance tests itself (32 per
// warp ballot; scalar loads of p_i(d_i), q_i(d_i)), so all CTAs stream the same row
// without waiting for one another.  Uniforms: the sampler's Philox stream of the
// row, round i for the test of draft i, round L for the final draw.
#include "fs_device.cuh"
#include "fs_host.h"

namespace fsd {

struct SpecArgs {
    const float* draft;         // [B, L, V]
    const int32_t* tokens;      // [B, L]
    const float* target;        // [B, L + 1, V]
    int L;
    int V;
    unsigned long long seed, offset;
    int32_t* out_tokens;        // [B, L + 1]
    int32_t* out_accepted;      // [B]
    int32_t* out_emitted;       // [B]
    int shift;
    int ns;
    int nsc;
};

template <bool VEC>
__global__ void __launch_bounds__(NT, 4) spec_kernel(const SpecArgs a) {
    const int C = int(cluster_nctarank());
    const int rank = int(cluster_ctarank());
    const int b = int(cluster_id_x());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool leader = rank == 0;
    const Smem sm(a.ns);
    Geom g(a.V, a.shift, a.ns, a.nsc, rank);
    const int V = a.V, L = a.L;
    grid_dependency_wait();
    allow_dependents();

    // ---- the chain: the first rejected draft (L when all are accepted)
    if (warp == 0) {
        int first = L;
#pragma unroll 1
        for (int i0 = 0; i0 < L; i0 += 32) {
            const int i = i0 + lane;
            bool rej = false;
            if (i < L) {
                const int d = a.tokens[size_t(b) * L + i];
                rej = true;  // a draft token outside the vocabulary is rejected
                if (d >= 0 && d < V) {
                    const float pd = a.target[(size_t(b) * (L + 1) + i) * size_t(V) + d];
                    const float qd = a.draft[(size_t(b) * L + i) * size_t(V) + d];
                    const float u = sampler_uniform(a.seed, a.offset, uint32_t(b), uint32_t(i));
                    rej = !(u * qd < pd);
                }
            }
            const unsigned bal = __ballot_sync(FULL, rej);
            if (bal) {
                first = i0 + __ffs(bal) - 1;
                break;
            }
        }
        if (lane == 0) sm.red()[100] = first;
    }
    __syncthreads();
    const int pos = sm.red()[100];
    const float* row = a.target + (size_t(b) * (L + 1) + pos) * size_t(V);
    if (pos < L) g.qrow = a.draft + (size_t(b) * L + pos) * size_t(V);

    // ---- the row of weights: one pass, masses into the leader
    if (tid == 0) *sm.ctr() = NW;
    __syncthreads();
    cluster_arrive();
    int npos = 0;
    bool bad = false;
    uint32_t kmax = 0;
    pass1<VEC, true, true>(row, g, sm, -1, warp, lane, npos, bad, kmax);
    cluster_wait();  // every CTA has started
    pass1_totals(g, sm, leader, rank, C, npos, bad, kmax, -1, true, true, warp, lane, tid);
    cluster_sync();  // the leader's segment table and every CTA's part are complete
    if (!leader) return;

    // ---- the draw (leader) and the outputs
    const Totals tot = cluster_totals(sm, C);
    if (tid < C) sm.cmass()[tid] = sm.part()[tid].f[0];
    __syncthreads();
    if (warp != 0) return;
    const bool valid = !tot.any_bad && tot.M > 0.f && tot.M <= 3.402823466e38f;
    int token = -1;
    if (valid) {
        const float u = sampler_uniform(a.seed, a.offset, uint32_t(b), uint32_t(L));
        token = unpack_j(draw_full<VEC>(row, g, sm, C, 0, 0.f, u * tot.M, lane));
    }
    for (int i = lane; i <= L; i += 32) {
        int v = -1;
        if (i < pos) v = a.tokens[size_t(b) * L + i];
        if (i == pos) v = token;
        a.out_tokens[size_t(b) * (L + 1) + i] = v;
    }
    if (lane == 0) {
        a.out_accepted[b] = pos;
        a.out_emitted[b] = pos + (token >= 0 ? 1 : 0);
    }
}

}  // namespace fsd

extern "C" {

fs_status fs_chain_speculative_sampling(const float* draft_probs, const int32_t* draft_tokens,
                                        const float* target_probs, int32_t batch, int32_t num_draft,
                                        int32_t vocab, uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                        int32_t* out_accepted, int32_t* out_emitted, void* stream) {
    using namespace fsd;
    if (batch < 0 || num_draft < 0 || vocab < 1) return FS_ERR_INVALID_ARG;
    if (batch == 0) return FS_OK;
    if (!target_probs || !out_tokens || !out_accepted || !out_emitted) return FS_ERR_INVALID_ARG;
    if (num_draft > 0 && (!draft_probs || !draft_tokens)) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    if (int64_t(batch) * (int64_t(num_draft) + 1) > int64_t(0x7fffffff)) return FS_ERR_UNSUPPORTED;
    const bool aligned = ((reinterpret_cast<uintptr_t>(target_probs) & 15) == 0) &&
                         (num_draft == 0 || (reinterpret_cast<uintptr_t>(draft_probs) & 15) == 0);
    const bool vec = (vocab % 4 == 0) && aligned;
    const void* fn = vec ? reinterpret_cast<const void*>(spec_kernel<true>)
                         : reinterpret_cast<const void*>(spec_kernel<false>);
    Plan p;
    fs_status st = make_plan(batch, vocab, fn, true, p);
    if (st != FS_OK) return st;
    SpecArgs a;
    a.draft = draft_probs;
    a.tokens = draft_tokens;
    a.target = target_probs;
    a.L = num_draft;
    a.V = vocab;
    a.seed = seed;
    a.offset = offset;
    a.out_tokens = out_tokens;
    a.out_accepted = out_accepted;
    a.out_emitted = out_emitted;
    a.shift = p.shift;
    a.ns = p.ns;
    a.nsc = p.nsc;
    if (vec) return launch_cluster(spec_kernel<true>, p, batch, stream, a);
    return launch_cluster(spec_kernel<false>, p, batch, stream, a);
}

}  // extern "C"
