// Cross-resource staggering of verification: phase planning, a discrete-event
// model of the KV_full staging ring, and draft-horizon sizing.  Host code.
//
// "VeriCache: Making Lossy KV Compression Exact", "Verifying Without Giving
// Back the Speedup" and Figure 2: requests do not all draft and then all
// verify; their verifications are spread over time, so the transfer of one
// request's full cache overlaps the drafting of the others.  Study notes
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", case 2
// (full KV on the CPU): stagger who verifies so that few full caches cross
// the link at once.  "VeriCache Guide", "The Amortized Drafting Horizon"
// (effective swap cost per token T_swap / L) and "Best Practice 1" (choose the
// horizon so that the swap ends before drafting does).
//
// Model.  Request r cycles through P = x + 1 ticks: it verifies at the ticks
// t with t mod P == phase[r] and drafts one token at every other tick.  A tick
// runs every layer in order; its compute time is the sum over its drafting
// requests of draft_ns[r] and over its verifying requests of verify_ns[r]
// (both for all layers), plus tick_ns.  The verifying requests of a tick form
// one staging job: their KV_full (stage_bytes, all layers) is copied over the
// link at link_bytes_per_ns into one of n_slots staging buffers, layer by
// layer.  The staging stream takes the jobs in tick order; a job starts when
// the previous job is done and its slot is free (the slot's previous job's
// tick has ended).  Layer l of a tick starts when layer l - 1 has ended and,
// if the tick verifies, when layer l of its job has landed; the difference is
// a stall.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "vc.h"

namespace {

struct Job {
    int64_t tick;
    double bytes;
};

// per-phase compute time (ns) and staging bytes of a plan
void phase_costs(const vc_stagger_model &m, int32_t n_phases, const int32_t *phase, std::vector<double> &tick_ns,
                 std::vector<double> &bytes) {
    double all_draft = 0.0;
    for (int r = 0; r < m.n_requests; ++r) all_draft += m.draft_ns[r];
    tick_ns.assign(n_phases, all_draft + m.tick_ns);
    bytes.assign(n_phases, 0.0);
    for (int r = 0; r < m.n_requests; ++r) {
        tick_ns[phase[r]] += m.verify_ns[r] - m.draft_ns[r];
        bytes[phase[r]] += (double)m.stage_bytes[r];
    }
}

bool model_ok(const vc_stagger_model *m) {
    if (!m || m->n_requests < 0 || m->n_slots < 1 || m->n_layers < 1 || !(m->link_bytes_per_ns > 0.0) ||
        !(m->tick_ns >= 0.0))
        return false;
    if (m->n_requests > 0 && (!m->stage_bytes || !m->draft_ns || !m->verify_ns)) return false;
    for (int r = 0; r < m->n_requests; ++r)
        if (m->stage_bytes[r] < 0 || !(m->draft_ns[r] >= 0.0) || !(m->verify_ns[r] >= 0.0)) return false;
    return true;
}

}  // namespace

extern "C" {

VC_API vc_status vc_stagger_plan(const int64_t *stage_bytes, int32_t n, int32_t n_phases, int32_t *phase,
                                 int64_t *phase_bytes) {
    if (n < 0 || n_phases < 1 || (n > 0 && (!stage_bytes || !phase))) return VC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r)
        if (stage_bytes[r] < 0) return VC_ERR_INVALID_ARG;
    // 1. longest processing time first into G = min(n, n_phases) groups:
    //    requests by decreasing bytes (ties to the lower index), each to the
    //    group holding the fewest bytes so far (ties to the lower group)
    const int G = std::max(1, std::min<int>(n, n_phases));
    std::vector<int> order(n);
    for (int r = 0; r < n; ++r) order[r] = r;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return stage_bytes[a] > stage_bytes[b]; });
    std::vector<int64_t> load(G, 0);
    std::vector<int> group(n, 0);
    for (int r : order) {
        int best = 0;
        for (int g = 1; g < G; ++g)
            if (load[g] < load[best]) best = g;
        group[r] = best;
        load[best] += stage_bytes[r];
    }
    // 2. groups by decreasing load (ties to the lower group), interleaved
    //    largest, smallest, second largest, ... so that a large job follows
    //    a small one and the link can run ahead of it
    std::vector<int> byload(G);
    for (int g = 0; g < G; ++g) byload[g] = g;
    std::stable_sort(byload.begin(), byload.end(), [&](int a, int b) { return load[a] > load[b]; });
    std::vector<int> seq;
    for (int lo = 0, hi = G - 1; lo <= hi; ++lo, --hi) {
        seq.push_back(byload[lo]);
        if (hi != lo) seq.push_back(byload[hi]);
    }
    // 3. the k-th group of that sequence verifies at phase floor(k P / G):
    //    evenly spaced over the cycle when there are fewer groups than phases
    std::vector<int> gphase(G);
    for (int k = 0; k < G; ++k) gphase[seq[k]] = (int)(((int64_t)k * n_phases) / G);
    for (int r = 0; r < n; ++r) phase[r] = gphase[group[r]];
    if (phase_bytes) {
        for (int p = 0; p < n_phases; ++p) phase_bytes[p] = 0;
        for (int g = 0; g < G; ++g) phase_bytes[gphase[g]] += load[g];
    }
    return VC_OK;
}

VC_API vc_status vc_stagger_simulate(const vc_stagger_model *m, int32_t n_phases, const int32_t *phase,
                                     int32_t n_cycles, vc_stagger_result *out) {
    if (!model_ok(m) || n_phases < 1 || n_cycles < 1 || !out || (m->n_requests > 0 && !phase))
        return VC_ERR_INVALID_ARG;
    for (int r = 0; r < m->n_requests; ++r)
        if (phase[r] < 0 || phase[r] >= n_phases) return VC_ERR_INVALID_ARG;
    std::vector<double> tick_ns, bytes;
    phase_costs(*m, n_phases, phase, tick_ns, bytes);
    const int L = m->n_layers;
    const double bw = m->link_bytes_per_ns;
    const int64_t n_ticks = (int64_t)n_phases * n_cycles;

    // staging jobs in tick order, with their per-layer landing times
    std::vector<Job> jobs;
    for (int64_t t = 0; t < n_ticks; ++t)
        if (bytes[t % n_phases] > 0.0) jobs.push_back({t, bytes[t % n_phases]});
    std::vector<double> tick_end(n_ticks, 0.0), job_end(jobs.size(), 0.0);
    std::vector<double> landed((size_t)jobs.size() * L, 0.0);
    std::vector<double> stall(n_ticks, 0.0);
    // Jobs and ticks are processed in tick order: job i depends on job i - 1
    // and on the tick of job i - n_slots (earlier than job i's own tick), so
    // every job a tick waits for is computed before the tick.
    size_t next_job = 0;
    double prev_end = 0.0;
    for (int64_t t = 0; t < n_ticks; ++t) {
        // schedule every job whose slot is freed by a tick before t (jobs
        // for tick t and later whose dependencies are known)
        while (next_job < jobs.size()) {
            const size_t i = next_job;
            double start = i > 0 ? job_end[i - 1] : 0.0;
            if (i >= (size_t)m->n_slots) {
                const int64_t ft = jobs[i - m->n_slots].tick;
                if (ft >= t) break;  // its slot is freed at a tick not yet computed
                start = std::max(start, tick_end[ft]);
            }
            const double per_layer = jobs[i].bytes / bw / L;
            for (int l = 0; l < L; ++l) landed[i * L + l] = start + per_layer * (l + 1);
            job_end[i] = start + jobs[i].bytes / bw;
            ++next_job;
        }
        const double per_layer = tick_ns[t % n_phases] / L;
        double clock = prev_end;
        const bool verifies = bytes[t % n_phases] > 0.0;
        size_t j = 0;
        if (verifies) {
            // the job of this tick (jobs are in tick order)
            j = (size_t)(std::lower_bound(jobs.begin(), jobs.end(), t,
                                          [](const Job &a, int64_t tt) { return a.tick < tt; }) -
                         jobs.begin());
        }
        for (int l = 0; l < L; ++l) {
            if (verifies) {
                // job j was scheduled: its slot's previous tick precedes t
                const double ready = landed[j * L + l];
                if (ready > clock) {
                    stall[t] += ready - clock;
                    clock = ready;
                }
            }
            clock += per_layer;
        }
        tick_end[t] = clock;
        prev_end = clock;
    }

    // steady-state figures over the last cycle
    const int64_t t0 = (int64_t)(n_cycles - 1) * n_phases;
    const double start = t0 > 0 ? tick_end[t0 - 1] : 0.0;
    double st = 0.0, comp = 0.0, stage = 0.0, maxb = 0.0;
    for (int64_t t = t0; t < n_ticks; ++t) {
        st += stall[t];
        comp += tick_ns[t % n_phases];
        stage += bytes[t % n_phases] / bw;
    }
    for (int p = 0; p < n_phases; ++p) maxb = std::max(maxb, bytes[p]);
    out->cycle_ns = tick_end[n_ticks - 1] - start;
    out->compute_ns = comp;
    out->stall_ns = st;
    out->stage_ns = stage;
    out->overlap = stage > 0.0 ? std::min(1.0, std::max(0.0, 1.0 - st / stage)) : 1.0;
    out->peak_stage_bytes = (int64_t)maxb * m->n_slots;
    out->draft_tokens_per_cycle = (int64_t)m->n_requests * (n_phases - 1);
    return VC_OK;
}

VC_API vc_status vc_stagger_horizon(const vc_stagger_model *m, int32_t x_lo, int32_t x_hi, int32_t n_cycles,
                                    int32_t *x_out, int32_t *phase, vc_stagger_result *out) {
    if (!model_ok(m) || x_lo < 1 || x_hi < x_lo || n_cycles < 1 || !x_out || !out ||
        (m->n_requests > 0 && !phase))
        return VC_ERR_INVALID_ARG;
    std::vector<int32_t> ph(std::max(1, m->n_requests));
    for (int32_t x = x_lo; x <= x_hi; ++x) {
        vc_status s = vc_stagger_plan(m->stage_bytes, m->n_requests, x + 1, ph.data(), nullptr);
        if (s != VC_OK) return s;
        vc_stagger_result r;
        s = vc_stagger_simulate(m, x + 1, ph.data(), n_cycles, &r);
        if (s != VC_OK) return s;
        // the smallest horizon whose steady state hides every staged byte
        if (r.stall_ns <= 0.0 || x == x_hi) {
            *x_out = x;
            *out = r;
            for (int i = 0; i < m->n_requests; ++i) phase[i] = ph[i];
            return VC_OK;
        }
    }
    return VC_ERR_INVALID_ARG;  // unreachable
}

}  // extern "C"

// the Python binding mirrors these layouts
static_assert(sizeof(vc_stagger_model) == 56, "vc_stagger_model layout");
static_assert(sizeof(vc_stagger_result) == 56, "vc_stagger_result layout");
