// C ABI of the speculative-pipeline-decoding library: validation, workspace layout,
// the step schedule (target rounds on the caller's stream, the draft module on a
// second stream joined before the LM head), CUDA-graph capture, polling and results.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

using namespace spd;

namespace {
thread_local std::string g_create_error;
constexpr int GRAPH_STEPS = 8;      // steps per captured graph (timing reads happen per graph)
constexpr int LM_GRID_MAX = 4096;
constexpr int PF_ROWS = 512;
constexpr int SM_BOUND = 256;       // SM count bound used for workspace sizing
}  // namespace

struct spd_handle {
    Plan h{};
    Plan *dP = nullptr;
    cudaStream_t s_user = nullptr;                 // caller's stream (may be the legacy default stream)
    cudaStream_t s_main = nullptr, s_pdm = nullptr; // own streams: target rounds, draft module
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_in = nullptr, ev_out = nullptr;
    cudaGraphExec_t g1 = nullptr, gN = nullptr;
    int grid_gemv = 0, grid_lm = 0, num_sms = 0;
    bool prefilled = false;
    std::string err;
    float theta = 1e4f;
    int use_graph = 0, timing = 0;
    std::vector<cudaEvent_t> tev;   // timing event pairs
    int tev_next = 0;
    double t_ms = 0.0;
    long long t_launches = 0;
    int *host_pinned = nullptr;     // [8] small readback buffer
    size_t ws_bytes = 0;
    void *ws = nullptr;
    int elem = 2;                   // bytes of a weight element
};

static int fail(spd_handle *H, int code, const std::string &msg) {
    if (H) H->err = msg;
    else g_create_error = msg;
    return code;
}

#define CK(H, x)                                                                                 \
    do {                                                                                         \
        cudaError_t e_ = (x);                                                                    \
        if (e_ != cudaSuccess) return fail(H, SPD_ECUDA, std::string(#x) + ": " + cudaGetErrorString(e_)); \
    } while (0)

// ---------------------------------------------------------------------------------
// workspace layout (bump allocation, 256-byte aligned); base == nullptr only sizes
struct Bump {
    char *base;
    size_t off = 0;
    template <typename T>
    T *take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

static int validate(const spd_dims *d, int Ls, const spd_config *c, std::string &why) {
    if (!d || !c) { why = "null dims/config"; return SPD_EINVAL; }
    if (d->dtype != SPD_F32 && d->dtype != SPD_BF16) { why = "dtype must be SPD_F32 or SPD_BF16"; return SPD_EINVAL; }
    if (d->L < 1 || d->L > SPD_MAX_LAYERS) { why = "L out of range"; return SPD_EINVAL; }
    if (d->Hq < 1 || d->Hkv < 1 || d->Hq % d->Hkv) { why = "need Hq % Hkv == 0"; return SPD_EINVAL; }
    const int G = d->Hq / d->Hkv;
    if (G > 8 || (G & (G - 1))) { why = "GQA group Hq/Hkv must be 1, 2, 4 or 8"; return SPD_EINVAL; }
    if (d->hd != 64 && d->hd != 128) { why = "head dim must be 64 or 128"; return SPD_EINVAL; }
    const int vec = d->dtype == SPD_BF16 ? 8 : 4;
    if (d->d % 64 || d->F % 64 || (d->Hq * d->hd) % 64) { why = "d, F and Hq*hd must be multiples of 64"; return SPD_EINVAL; }
    if (d->d % vec || d->F % vec) { why = "bad vector width"; return SPD_EINVAL; }
    if (d->V < 2) { why = "V < 2"; return SPD_EINVAL; }
    if (!(d->rms_eps > 0.f) || !(d->rope_theta > 1.f)) { why = "rms_eps > 0 and rope_theta > 1 required"; return SPD_EINVAL; }
    if (c->n < 1 || c->n > SPD_MAX_STAGES || c->n > d->L) { why = "need 1 <= n <= min(L, 31)"; return SPD_EINVAL; }
    if (c->n_anchors < 1 || c->n_anchors > SPD_MAX_ANCHORS) { why = "n_anchors out of range"; return SPD_EINVAL; }
    if (c->anchors[0] != 0) { why = "anchors[0] must be 0 (the embedding)"; return SPD_EINVAL; }
    for (int i = 1; i < c->n_anchors; ++i)
        if (c->anchors[i] <= c->anchors[i - 1] || c->anchors[i] > d->L) { why = "anchors must increase within [0, L]"; return SPD_EINVAL; }
    if (Ls < 0 || Ls > SPD_MAX_PDM_LAYERS) { why = "Ls out of range"; return SPD_EINVAL; }
    if (c->max_new < 1) { why = "max_new < 1"; return SPD_EINVAL; }
    if (c->max_seq < c->max_new + c->n + 1) { why = "max_seq too small"; return SPD_EINVAL; }
    if (c->max_seq > 16384) { why = "max_seq above 16384 (attention merges at most 128 chunks)"; return SPD_EINVAL; }
    if (!(c->temperature >= 0.f)) { why = "temperature < 0"; return SPD_EINVAL; }
    if (c->force_p >= 0.f) {
        if (c->force_p > 1.f) { why = "force_p > 1"; return SPD_EINVAL; }
        if (c->temperature > 0.f) { why = "forced drafts are defined for T = 0 only"; return SPD_EINVAL; }
    }
    if (c->temperature > 0.f && Ls == 0) { why = "sampling needs a draft module"; return SPD_EINVAL; }
    if (c->speculate != SPD_SPEC_INPUT && c->speculate != SPD_SPEC_OUTPUT) {
        why = "speculate must be SPD_SPEC_INPUT or SPD_SPEC_OUTPUT";
        return SPD_EINVAL;
    }
    bool explicit_bounds = false;
    for (int s = 0; s <= SPD_MAX_STAGES; ++s) explicit_bounds = explicit_bounds || c->stage_bounds[s] != 0;
    if (explicit_bounds) {
        bool ok = c->stage_bounds[0] == 0 && c->stage_bounds[c->n] == d->L;
        for (int s = 0; s < c->n; ++s) ok = ok && c->stage_bounds[s + 1] > c->stage_bounds[s];
        for (int s = c->n + 1; s <= SPD_MAX_STAGES; ++s) ok = ok && c->stage_bounds[s] == 0;
        if (!ok) { why = "stage_bounds must be 0 = b_0 < b_1 < ... < b_n = L (zero past b_n)"; return SPD_EINVAL; }
    }
    return SPD_OK;
}

// Stage s holds layers [b[s], b[s + 1]): the caller's explicit bounds, else floor(s L / n).
static void stage_plan(const spd_dims *d, const spd_config *c, int *b) {
    bool explicit_bounds = false;
    for (int s = 0; s <= SPD_MAX_STAGES; ++s) explicit_bounds = explicit_bounds || c->stage_bounds[s] != 0;
    for (int s = 0; s <= c->n; ++s) b[s] = explicit_bounds ? c->stage_bounds[s] : (int)(((long long)s * d->L) / c->n);
}

static size_t layout(const spd_dims *d, int Ls, const spd_config *c, char *base, Plan &h) {
    Bump b{base};
    const int n = c->n, ns = n + 1, elem = (int)sizeof(KvT<float>);   // KV cache elements (fp32)
    const int qkv = (d->Hq + 2 * d->Hkv) * d->hd, qr = d->Hq * d->hd;
    const int max_chunks = (c->max_seq + ATT_CHUNK - 1) / ATT_CHUNK;
    const int max_steps = n * c->max_new + 2 * n + 8;
    const long long kvs = (long long)c->max_seq * d->Hkv * d->hd;
    h.st = b.take<DevState>(1);
    h.X = b.take<float>((size_t)ns * d->d);
    h.QKV = b.take<float>((size_t)n * qkv);
    h.U = b.take<float>((size_t)n * 2 * d->F);
    h.ANCH = b.take<float>((size_t)ns * c->n_anchors * d->d);
    h.kc = b.take<char>((size_t)d->L * kvs * elem);
    h.vc = b.take<char>((size_t)d->L * kvs * elem);
    h.pkc = b.take<char>((size_t)std::max(Ls, 1) * kvs * elem);
    h.pvc = b.take<char>((size_t)std::max(Ls, 1) * kvs * elem);
    h.rope = b.take<float2>((size_t)c->max_seq * (d->hd / 2));
    h.att_part = b.take<float>((size_t)MAXS * d->Hq * max_chunks * (d->hd + 4));
    h.patt_part = b.take<float>((size_t)MAXS * d->Hq * max_chunks * (d->hd + 4));
    h.att_cnt = b.take<int>((size_t)MAXS * d->Hkv);
    h.patt_cnt = b.take<int>((size_t)MAXS * d->Hkv);
    h.Xp = b.take<float>((size_t)ns * d->d);
    h.QKVp = b.take<float>((size_t)ns * qkv);
    h.ATTp = b.take<float>((size_t)ns * qr);
    h.GUp = b.take<float>((size_t)ns * d->F);
    // bf16 input rows of the draft GEMMs: hi parts, then lo parts of the same size
    h.Xb = b.take<__nv_bfloat16>((size_t)2 * ns * d->d);
    h.ATTb = b.take<__nv_bfloat16>((size_t)2 * ns * qr);
    h.GUb = b.take<__nv_bfloat16>((size_t)2 * ns * d->F);
    h.Xlm = b.take<__nv_bfloat16>((size_t)4 * d->d);
    h.ANCHb = b.take<__nv_bfloat16>((size_t)2 * ns * c->n_anchors * d->d);
    h.ssp = b.take<float>((size_t)MAXS * (d->d / 8));
    {
        // draft GEMM K-slab partials: largest slabs x rows x outputs over the five GEMMs
        int kx[6], nsl[6], MT;
        pdm_plan(d->d, d->F, qr, c->n_anchors, n, d->dtype, kx, nsl, &MT);
        const int Ns[5] = {d->d, qkv, d->d, 2 * d->F, d->d};
        size_t most = 1;
        for (int i = 0; i < 5; ++i)
            if (nsl[i] > 1) most = std::max(most, (size_t)nsl[i] * ns * Ns[i]);
        h.pdm_part = b.take<float>(most);
        h.pdm_cnt = b.take<int>((size_t)SM_BOUND);
    }
    h.logits = b.take<float>((size_t)2 * d->V);
    h.dlogits = b.take<float>(c->temperature > 0.f ? (size_t)ns * d->V : 1);
    h.lm_part = b.take<float>((size_t)LM_GRID_MAX * 4);
    h.lm_stat = b.take<float>((size_t)LM_GRID_MAX * 4);
    h.lm_cnt = b.take<int>(1);
    h.trace = b.take<spd_trace_rec>((size_t)max_steps);
    h.trace_len = b.take<int>((size_t)max_steps * d->L);
    h.out_tokens = b.take<int>((size_t)c->max_new);
    h.pf_rows = PF_ROWS;
    h.pf_H = b.take<float>((size_t)PF_ROWS * d->d);
    h.pf_XN = b.take<float>((size_t)PF_ROWS * std::max(d->d, d->F));
    h.pf_QKV = b.take<float>((size_t)PF_ROWS * qkv);
    h.pf_ATT = b.take<float>((size_t)PF_ROWS * qr);
    h.pf_GU = b.take<float>((size_t)PF_ROWS * 2 * d->F);
    h.pf_ANCH = b.take<float>((size_t)PF_ROWS * c->n_anchors * d->d);
    h.pf_Hp = b.take<float>((size_t)PF_ROWS * d->d);
    h.pf_logits = b.take<float>((size_t)d->V);
    {
        const int kmax = std::max(std::max(d->d, d->F), std::max(qr, c->n_anchors * d->d));
        h.pf_A2 = b.take<__nv_bfloat16>(d->dtype == SPD_BF16 ? (size_t)2 * PF_ROWS * kmax : 1);
    }
    Plan *dp = b.take<Plan>(1);
    h.self = dp;
    h.kv_stride = kvs;
    h.att_max_chunks = max_chunks;
    h.max_steps = max_steps;
    return b.off + 256;
}

extern "C" int spd_workspace_bytes(const spd_dims *d, const spd_pdm_weights *pw, const spd_config *c, size_t *bytes) {
    std::string why;
    const int Ls = pw ? pw->Ls : 0;
    if (!bytes) return fail(nullptr, SPD_EINVAL, "bytes is NULL");
    const int rc = validate(d, Ls, c, why);
    if (rc) return fail(nullptr, rc, why);
    Plan tmp{};
    *bytes = layout(d, Ls, c, nullptr, tmp);
    return SPD_OK;
}

// ---------------------------------------------------------------------------------
template <typename T>
static void record_step(spd_handle *H, std::vector<int> *pairs) {
    const Plan &h = H->h;
    Plan *P = H->dP;
    // input-state schedule: the draft module on the second stream, concurrent with the
    // target's rounds; output-state schedule: on the target's stream after its rounds
    const bool separate = h.Ls > 0 && !h.spec_out;
    if (separate) {
        cudaEventRecord(H->ev_fork, H->s_main);
        cudaStreamWaitEvent(H->s_pdm, H->ev_fork, 0);
        launch_pdm_step<T>(P, h, H->num_sms, H->s_pdm);
        cudaEventRecord(H->ev_join, H->s_pdm);
    }
    for (int j = 0; j < h.J; ++j) {
        launch_target_qkv<T>(P, h, j, H->grid_gemv, H->s_main);
        launch_target_attn<T>(P, h, j, H->s_main);
        launch_target_oproj<T>(P, h, j, H->grid_gemv, H->s_main);
        int pi = -1;
        if (pairs) {
            pi = H->tev_next;
            H->tev_next += 2;
            cudaEventRecordWithFlags(H->tev[pi], H->s_main, cudaEventRecordExternal);
        }
        launch_target_gateup<T>(P, h, j, H->grid_gemv, H->s_main);
        if (pairs) {
            cudaEventRecordWithFlags(H->tev[pi + 1], H->s_main, cudaEventRecordExternal);
            pairs->push_back(pi);
        }
        launch_target_down<T>(P, h, j, H->grid_gemv, H->s_main);
    }
    if (separate) cudaStreamWaitEvent(H->s_main, H->ev_join, 0);
    if (h.Ls > 0 && h.spec_out) launch_pdm_step<T>(P, h, H->num_sms, H->s_main);
    launch_lm_head<T>(P, h, H->grid_lm, H->s_main);
    launch_verify<T>(P, h, H->s_main);
}

static void record_step_any(spd_handle *H, std::vector<int> *pairs) {
    if (H->h.dtype == SPD_BF16) record_step<__nv_bfloat16>(H, pairs);
    else record_step<float>(H, pairs);
}

static int capture(spd_handle *H, int steps, cudaGraphExec_t *out, std::vector<int> *pairs) {
    cudaGraph_t g = nullptr;
    CK(H, cudaStreamBeginCapture(H->s_main, cudaStreamCaptureModeThreadLocal));
    for (int i = 0; i < steps; ++i) record_step_any(H, pairs);
    CK(H, cudaStreamEndCapture(H->s_main, &g));
    CK(H, cudaGraphInstantiate(out, g, 0));
    cudaGraphDestroy(g);
    return SPD_OK;
}

struct HandleTiming {
    std::vector<int> p1, pN;
};

static HandleTiming &timing_of(spd_handle *H) {
    static thread_local std::vector<std::pair<spd_handle *, HandleTiming>> tab;
    for (auto &e : tab)
        if (e.first == H) return e.second;
    tab.emplace_back(H, HandleTiming{});
    return tab.back().second;
}

extern "C" int spd_create(const spd_dims *d, const spd_target_weights *tw, const spd_pdm_weights *pw,
                          const spd_config *c, void *workspace, size_t ws_bytes, void *stream, spd_handle **out) {
    if (!out) return fail(nullptr, SPD_EINVAL, "out is NULL");
    *out = nullptr;
    std::string why;
    const int Ls = pw ? pw->Ls : 0;
    int rc = validate(d, Ls, c, why);
    if (rc) return fail(nullptr, rc, why);
    if (!tw || !tw->embed || !tw->layers || !tw->final_norm || !tw->lm_head) return fail(nullptr, SPD_EINVAL, "null target weights");
    for (int l = 0; l < d->L; ++l) {
        const spd_layer_weights &w = tw->layers[l];
        if (!w.wq || !w.wk || !w.wv || !w.wo || !w.w_gate || !w.w_up || !w.w_down || !w.attn_norm || !w.ffn_norm)
            return fail(nullptr, SPD_EINVAL, "null pointer in target layer " + std::to_string(l));
    }
    if (Ls > 0) {
        if (!pw->proj || !pw->layers || !pw->final_norm || !pw->lm_head) return fail(nullptr, SPD_EINVAL, "null draft weights");
        for (int l = 0; l < Ls; ++l) {
            const spd_layer_weights &w = pw->layers[l];
            if (!w.wq || !w.wk || !w.wv || !w.wo || !w.w_gate || !w.w_up || !w.w_down || !w.attn_norm || !w.ffn_norm)
                return fail(nullptr, SPD_EINVAL, "null pointer in draft layer " + std::to_string(l));
        }
    }
    // weight matrices are streamed with 16-byte bulk copies and loads
    auto a16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    auto layer_ok = [&](const spd_layer_weights &w) {
        return a16(w.wq) && a16(w.wk) && a16(w.wv) && a16(w.wo) && a16(w.w_gate) && a16(w.w_up) && a16(w.w_down) &&
               a16(w.attn_norm) && a16(w.ffn_norm);
    };
    bool aligned = a16(tw->embed) && a16(tw->lm_head) && a16(tw->final_norm);
    for (int l = 0; l < d->L; ++l) aligned = aligned && layer_ok(tw->layers[l]);
    if (Ls > 0) {
        aligned = aligned && a16(pw->proj) && a16(pw->lm_head) && a16(pw->final_norm);
        for (int l = 0; l < Ls; ++l) aligned = aligned && layer_ok(pw->layers[l]);
    }
    if (!aligned) return fail(nullptr, SPD_EINVAL, "weight pointers must be 16-byte aligned");
    if (c->force_p >= 0.f && (!c->forced_ref || c->forced_ref_len < 1)) return fail(nullptr, SPD_EINVAL, "forced drafts need forced_ref");
    if (!workspace) return fail(nullptr, SPD_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(nullptr, SPD_EINVAL, "workspace must be 256-byte aligned");
    Plan tmp{};
    const size_t need = layout(d, Ls, c, nullptr, tmp);
    if (ws_bytes < need) return fail(nullptr, SPD_ENOMEM, "workspace too small: need " + std::to_string(need));

    spd_handle *H = new spd_handle();
    Plan &h = H->h;
    layout(d, Ls, c, reinterpret_cast<char *>(workspace), h);
    H->dP = h.self;
    H->ws = workspace;
    H->ws_bytes = ws_bytes;
    H->elem = d->dtype == SPD_BF16 ? 2 : 4;
    h.L = d->L; h.d = d->d; h.Hq = d->Hq; h.Hkv = d->Hkv; h.hd = d->hd; h.F = d->F; h.V = d->V;
    h.n = c->n; h.nB = c->n_anchors; h.Ls = Ls; h.max_seq = c->max_seq; h.max_new = c->max_new; h.dtype = d->dtype;
    h.q_rows = d->Hq * d->hd; h.kv_rows = d->Hkv * d->hd; h.qkv_rows = h.q_rows + 2 * h.kv_rows;
    h.J = 0;
    stage_plan(d, c, h.b);
    for (int s = 0; s < c->n; ++s) h.J = std::max(h.J, h.b[s + 1] - h.b[s]);
    h.spec_out = c->speculate == SPD_SPEC_OUTPUT ? 1 : 0;
    for (int a = 0; a <= SPD_MAX_LAYERS; ++a) h.aidx[a] = -1;
    for (int i = 0; i < c->n_anchors; ++i) {
        h.anchors[i] = c->anchors[i];
        h.aidx[c->anchors[i]] = (signed char)i;
    }
    h.eps = d->rms_eps;
    h.scale = 1.0f / std::sqrt((float)d->hd);
    h.temperature = c->temperature;
    h.seed_lo = (unsigned)(c->seed & 0xffffffffull);
    h.seed_hi = (unsigned)(c->seed >> 32);
    h.forced = c->force_p >= 0.f;
    h.forced_thr = h.forced ? (unsigned)std::ceil((double)c->force_p * 16777216.0) : 0u;
    h.forced_ref = c->forced_ref;
    h.forced_ref_len = c->forced_ref_len;
    h.embed = tw->embed;
    h.lm_head = tw->lm_head;
    h.gf = tw->final_norm;
    for (int l = 0; l < d->L; ++l) {
        const spd_layer_weights &w = tw->layers[l];
        h.tl[l] = LayerW{w.wq, w.wk, w.wv, w.wo, w.w_gate, w.w_up, w.w_down, w.attn_norm, w.ffn_norm};
    }
    if (Ls > 0) {
        h.proj = pw->proj;
        h.pdm_gf = pw->final_norm;
        h.pdm_lm_head = pw->lm_head;
        for (int l = 0; l < Ls; ++l) {
            const spd_layer_weights &w = pw->layers[l];
            h.pl[l] = LayerW{w.wq, w.wk, w.wv, w.wo, w.w_gate, w.w_up, w.w_down, w.attn_norm, w.ffn_norm};
        }
    } else {
        h.proj = nullptr;
        h.pdm_gf = tw->final_norm;
        h.pdm_lm_head = tw->lm_head;
    }
    const long long el = H->elem;
    h.layer_bytes = el * ((long long)h.qkv_rows * h.d + (long long)h.d * h.q_rows + 3LL * h.F * h.d);
    h.pdm_bytes = Ls > 0 ? el * ((long long)h.d * h.nB * h.d + (long long)Ls * (h.layer_bytes / el)) : 0;
    h.lm_bytes = el * (long long)h.V * h.d * ((Ls > 0 && h.pdm_lm_head != h.lm_head) ? 2 : 1);
    H->theta = d->rope_theta;
    H->use_graph = c->graph;
    H->timing = c->timing;
    H->s_user = reinterpret_cast<cudaStream_t>(stream);

    auto bail = [&](int code) {
        g_create_error = H->err;
        spd_destroy(H);
        return code;
    };
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&H->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        H->err = "no CUDA device";
        return bail(SPD_ECUDA);
    }
    pdm_plan(h.d, h.F, h.q_rows, h.nB, h.n, h.dtype, h.pdm_kx, h.pdm_ns, &h.pdm_MT);
    h.pdl = 1;
    // Test hooks for the bounded waits, read once here and off unless set:
    // SPD_TEST_WAIT_CYCLES=<n> bounds the grouped GEMV's mbarrier waits at n SM cycles instead
    // of about 2 s; SPD_TEST_WITHHOLD_TILE=1 makes the first step's first gate/up launch skip
    // loading one tile, so a wait runs out and the step reports SPD_EDEVICE (ERR_TIMEOUT).
    h.wait_cycles = WAIT_LIMIT_CYCLES;
    h.test_withhold = 0;
    if (const char *e = std::getenv("SPD_TEST_WAIT_CYCLES")) {
        const long long v = std::atoll(e);
        if (v > 0) h.wait_cycles = v;
    }
    if (const char *e = std::getenv("SPD_TEST_WITHHOLD_TILE")) h.test_withhold = std::atoi(e) == 1 ? 1 : 0;
    const int gsm = gemv_smem_bytes(h);
    set_target_attributes(std::max(gsm, 48 * 1024));
    set_pdm_attributes();
    set_prefill_attributes();
    set_attn_attributes();
    H->num_sms = std::min(H->num_sms, SM_BOUND);
    H->grid_gemv = H->num_sms * target_blocks_per_sm(h.dtype, gemv_smem_bytes(h));
    H->grid_lm = std::min(LM_GRID_MAX, H->num_sms * lm_blocks_per_sm(h.dtype, 2 * h.d * 4, h.pdm_lm_head == h.lm_head));
    h.lm_stats = (lm_on_tensor_cores(h) && h.temperature > 0.f) ? 1 : 0;
    if (cudaStreamCreateWithFlags(&H->s_main, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&H->s_pdm, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&H->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&H->ev_join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&H->ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&H->ev_out, cudaEventDisableTiming) != cudaSuccess ||
        cudaMallocHost(&H->host_pinned, 64) != cudaSuccess) {
        H->err = "stream/event creation failed";
        return bail(SPD_ECUDA);
    }
    if (H->timing) {
        const int pairs_per_step = h.J;
        H->tev.resize((size_t)2 * pairs_per_step * (GRAPH_STEPS + 1 + 1));
        for (auto &e : H->tev)
            if (cudaEventCreate(&e) != cudaSuccess) { H->err = "event creation failed"; return bail(SPD_ECUDA); }
    }
    // zero counters and state, build the RoPE table, upload the plan
    if (cudaMemsetAsync(workspace, 0, (char *)h.kc - (char *)workspace, H->s_main) != cudaSuccess ||
        cudaMemsetAsync(h.att_cnt, 0, sizeof(int) * MAXS * h.Hkv, H->s_main) != cudaSuccess ||
        cudaMemsetAsync(h.patt_cnt, 0, sizeof(int) * MAXS * h.Hkv, H->s_main) != cudaSuccess ||
        cudaMemsetAsync(h.pdm_cnt, 0, sizeof(int) * SM_BOUND, H->s_main) != cudaSuccess ||
        cudaMemsetAsync(h.lm_cnt, 0, sizeof(int), H->s_main) != cudaSuccess ||
        cudaMemsetAsync(h.Xlm, 0, sizeof(__nv_bfloat16) * 4 * h.d, H->s_main) != cudaSuccess) {
        H->err = "workspace initialisation failed";
        return bail(SPD_ECUDA);
    }
    launch_rope_table(h, H->theta, H->s_main);
    if (cudaMemcpyAsync(H->dP, &h, sizeof(Plan), cudaMemcpyHostToDevice, H->s_main) != cudaSuccess ||
        cudaStreamSynchronize(H->s_main) != cudaSuccess) {
        H->err = std::string("plan upload failed: ") + cudaGetErrorString(cudaGetLastError());
        return bail(SPD_ECUDA);
    }
    if (cudaGetLastError() != cudaSuccess) {
        H->err = "kernel launch failed during create";
        return bail(SPD_ECUDA);
    }
    *out = H;
    return SPD_OK;
}

// Work of a call is ordered after everything already queued on the caller's stream, and
// the caller's stream is ordered after the call's work.
static int enter(spd_handle *H) {
    CK(H, cudaEventRecord(H->ev_in, H->s_user));
    CK(H, cudaStreamWaitEvent(H->s_main, H->ev_in, 0));
    return SPD_OK;
}
static int leave(spd_handle *H) {
    CK(H, cudaEventRecord(H->ev_out, H->s_main));
    CK(H, cudaStreamWaitEvent(H->s_user, H->ev_out, 0));
    return SPD_OK;
}

extern "C" int spd_prefill(spd_handle *H, const int32_t *prompt, int32_t prompt_len) {
    if (!H) return SPD_EINVAL;
    if (!prompt || prompt_len < 1) return fail(H, SPD_EINVAL, "empty prompt");
    if ((long long)prompt_len + H->h.max_new + H->h.n > H->h.max_seq)
        return fail(H, SPD_ECAPACITY, "prompt_len + max_new + n exceeds max_seq");
    int rc = enter(H);
    if (rc) return rc;
    const int enc = H->h.dtype == SPD_BF16
                        ? launch_prefill<__nv_bfloat16>(H->dP, H->h, prompt, prompt_len, H->num_sms, H->s_main)
                        : launch_prefill<float>(H->dP, H->h, prompt, prompt_len, H->num_sms, H->s_main);
    const cudaError_t le = cudaGetLastError();
    rc = leave(H);
    if (enc) return fail(H, SPD_ECUDA, "prefill: a TMA tensor map could not be encoded");
    if (le != cudaSuccess) return fail(H, SPD_ECUDA, std::string("prefill launch: ") + cudaGetErrorString(le));
    if (rc) return rc;
    H->prefilled = true;
    H->t_ms = 0.0;
    H->t_launches = 0;
    return SPD_OK;
}

static int read_state(spd_handle *H, int *N, int *done, int *error) {
    CK(H, cudaMemcpyAsync(H->host_pinned, H->h.st, 8 * sizeof(int), cudaMemcpyDeviceToHost, H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    if (N) *N = H->host_pinned[2];
    if (done) *done = H->host_pinned[3];
    if (error) *error = H->host_pinned[5];
    return SPD_OK;
}

static int collect_timing(spd_handle *H, const std::vector<int> &pairs) {
    for (int pi : pairs) {
        float ms = 0.f;
        CK(H, cudaEventSynchronize(H->tev[pi + 1]));
        CK(H, cudaEventElapsedTime(&ms, H->tev[pi], H->tev[pi + 1]));
        H->t_ms += ms;
        H->t_launches += 1;
    }
    return SPD_OK;
}

static int run_steps(spd_handle *H, int n_steps) {
    HandleTiming &ht = timing_of(H);
    if (H->use_graph) {
        if (!H->g1) {
            H->tev_next = 0;
            int rc = capture(H, 1, &H->g1, H->timing ? &ht.p1 : nullptr);
            if (rc) return rc;
            rc = capture(H, GRAPH_STEPS, &H->gN, H->timing ? &ht.pN : nullptr);
            if (rc) return rc;
        }
        int left = n_steps;
        while (left > 0) {
            const bool big = left >= GRAPH_STEPS;
            CK(H, cudaGraphLaunch(big ? H->gN : H->g1, H->s_main));
            left -= big ? GRAPH_STEPS : 1;
            if (H->timing) {
                const int rc = collect_timing(H, big ? ht.pN : ht.p1);
                if (rc) return rc;
            }
        }
    } else {
        for (int i = 0; i < n_steps; ++i) {
            std::vector<int> pairs;
            if (H->timing) H->tev_next = 0;
            record_step_any(H, H->timing ? &pairs : nullptr);
            if (H->timing) {
                const int rc = collect_timing(H, pairs);
                if (rc) return rc;
            }
        }
    }
    CK(H, cudaGetLastError());
    return SPD_OK;
}

extern "C" int spd_step(spd_handle *H, int32_t n_steps, int32_t *committed_host) {
    if (!H) return SPD_EINVAL;
    if (!H->prefilled) return fail(H, SPD_ESTATE, "spd_step before spd_prefill");
    if (n_steps < 0) return fail(H, SPD_EINVAL, "n_steps < 0");
    int rc = enter(H);
    if (rc) return rc;
    rc = run_steps(H, n_steps);
    if (rc) {
        const std::string keep = H->err;
        leave(H);
        H->err = keep;
        return rc;
    }
    rc = leave(H);
    if (rc) return rc;
    if (committed_host) {
        int N = 0, err = 0;
        rc = read_state(H, &N, nullptr, &err);
        if (rc) return rc;
        *committed_host = 1 + N;
        if (err) return fail(H, SPD_EDEVICE, "device error flag " + std::to_string(err));
    }
    return SPD_OK;
}

extern "C" int spd_get_stats(spd_handle *H, spd_stats *out) {
    if (!H || !out) return SPD_EINVAL;
    DevState st;
    CK(H, cudaMemcpyAsync(&st, H->h.st, sizeof(DevState), cudaMemcpyDeviceToHost, H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    std::memset(out, 0, sizeof(*out));
    out->N = st.N;
    out->K = st.t;
    out->accepts = st.accepts;
    out->rejects = st.rejects;
    out->alpha = st.t ? (double)st.N / st.t : 0.0;
    out->S0 = out->alpha * H->h.n;
    out->mean_kept_run = st.run_count ? (double)st.run_sum / st.run_count : (double)st.run_cur;
    out->weight_bytes = st.weight_bytes;
    out->ls_exceeds_masking = H->h.Ls > H->h.L / H->h.n ? 1 : 0;
    out->device_error = st.error;
    return SPD_OK;
}

extern "C" int spd_generate(spd_handle *H, const int32_t *prompt, int32_t prompt_len, int32_t on_host, int32_t *out_tokens,
                            int32_t *n_out_host, spd_stats *stats_host) {
    if (!H) return SPD_EINVAL;
    if (!prompt || !out_tokens) return fail(H, SPD_EINVAL, "null prompt/out");
    if (on_host && (prompt_len < 1 || (size_t)prompt_len > (size_t)H->h.max_steps * H->h.L))
        return fail(H, SPD_ECAPACITY, "prompt too long for host staging");
    const int32_t *pdev = prompt;
    int rc = enter(H);
    if (rc) return rc;
    // every exit after enter() orders the caller's stream after the work issued so far
    auto finish = [&](int code) {
        const std::string keep = H->err;
        const int lrc = leave(H);
        if (code) {
            H->err = keep;
            return code;
        }
        return lrc;
    };
    if (on_host) {
        // the prompt is staged in the per-step KV-length trace, unused until the first step
        const cudaError_t e = cudaMemcpyAsync(H->h.trace_len, prompt, (size_t)prompt_len * sizeof(int),
                                              cudaMemcpyHostToDevice, H->s_main);
        if (e != cudaSuccess) return finish(fail(H, SPD_ECUDA, std::string("prompt copy: ") + cudaGetErrorString(e)));
        pdev = H->h.trace_len;
    }
    rc = spd_prefill(H, pdev, prompt_len);
    if (rc) return finish(rc);
    const int max_new = H->h.max_new;
    int N = 0, done = 0, err = 0;
    rc = read_state(H, &N, &done, &err);
    if (rc) return finish(rc);
    long long issued = 0;
    while (!done && 1 + N < max_new) {
        if (issued >= H->h.max_steps) return finish(fail(H, SPD_EDEVICE, "no progress within the step bound"));
        int left = max_new - (1 + N);
        int k = left >= GRAPH_STEPS ? GRAPH_STEPS : left;
        rc = run_steps(H, k);
        if (rc) return finish(rc);
        issued += k;
        rc = read_state(H, &N, &done, &err);
        if (rc) return finish(rc);
        if (err) return finish(fail(H, SPD_EDEVICE, "device error flag " + std::to_string(err)));
    }
    cudaError_t e = cudaMemcpyAsync(out_tokens, H->h.out_tokens, (size_t)max_new * sizeof(int),
                                    on_host ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice, H->s_main);
    if (e == cudaSuccess) e = cudaStreamSynchronize(H->s_main);
    if (e != cudaSuccess) return finish(fail(H, SPD_ECUDA, std::string("token copy: ") + cudaGetErrorString(e)));
    rc = finish(SPD_OK);
    if (rc) return rc;
    if (n_out_host) *n_out_host = 1 + N;
    if (stats_host) return spd_get_stats(H, stats_host);
    return SPD_OK;
}

extern "C" int spd_get_trace(spd_handle *H, spd_trace_rec *recs, int32_t max_recs, int32_t *len_host, int32_t *count_host) {
    if (!H) return SPD_EINVAL;
    int t = 0;
    CK(H, cudaMemcpyAsync(H->host_pinned, &H->h.st->t, sizeof(int), cudaMemcpyDeviceToHost, H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    t = std::min(H->host_pinned[0], H->h.max_steps);
    const int k = std::min(t, std::max(0, max_recs));
    if (recs && k) CK(H, cudaMemcpy(recs, H->h.trace, (size_t)k * sizeof(spd_trace_rec), cudaMemcpyDeviceToHost));
    if (len_host && k) CK(H, cudaMemcpy(len_host, H->h.trace_len, (size_t)k * H->h.L * sizeof(int), cudaMemcpyDeviceToHost));
    if (count_host) *count_host = t;
    return SPD_OK;
}

extern "C" int spd_get_trace_view(spd_handle *H, spd_trace_view *out) {
    if (!H || !out) return SPD_EINVAL;
    CK(H, cudaMemcpyAsync(H->host_pinned, &H->h.st->t, sizeof(int), cudaMemcpyDeviceToHost, H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    out->recs = H->h.trace;
    out->kv_len = H->h.trace_len;
    out->count = std::min(H->host_pinned[0], H->h.max_steps);
    out->L = H->h.L;
    return SPD_OK;
}

extern "C" int spd_get_tokens(spd_handle *H, int32_t *tokens, int32_t max_tokens, int32_t *count_host) {
    if (!H || !tokens) return SPD_EINVAL;
    int N = 0;
    int rc = read_state(H, &N, nullptr, nullptr);
    if (rc) return rc;
    const int k = std::min(std::min(1 + N, H->h.max_new), max_tokens);
    if (k > 0) CK(H, cudaMemcpy(tokens, H->h.out_tokens, (size_t)k * sizeof(int), cudaMemcpyDeviceToHost));
    if (count_host) *count_host = 1 + N;
    return SPD_OK;
}

extern "C" int spd_read_buffer(spd_handle *H, int32_t which, int32_t index, size_t offset, void *dst, size_t bytes) {
    if (!H || !dst) return SPD_EINVAL;
    const Plan &h = H->h;
    const char *src = nullptr;
    size_t size = 0;
    const size_t kvb = (size_t)h.kv_stride * sizeof(KvT<float>);   // one layer's cache (fp32 rows)
    switch (which) {
        case SPD_BUF_RESIDUAL: src = (const char *)h.X; size = (size_t)(h.n + 1) * h.d * 4; break;
        case SPD_BUF_ANCHORS: src = (const char *)h.ANCH; size = (size_t)(h.n + 1) * h.nB * h.d * 4; break;
        case SPD_BUF_LOGITS: src = (const char *)h.logits; size = (size_t)2 * h.V * 4; break;
        case SPD_BUF_KCACHE:
        case SPD_BUF_VCACHE:
            if (index < 0 || index >= h.L) return fail(H, SPD_EINVAL, "layer index out of range");
            src = (const char *)(which == SPD_BUF_KCACHE ? h.kc : h.vc) + (size_t)index * kvb;
            size = kvb;
            break;
        case SPD_BUF_PDM_KCACHE:
        case SPD_BUF_PDM_VCACHE:
            if (index < 0 || index >= h.Ls) return fail(H, SPD_EINVAL, "draft layer index out of range");
            src = (const char *)(which == SPD_BUF_PDM_KCACHE ? h.pkc : h.pvc) + (size_t)index * kvb;
            size = kvb;
            break;
        case SPD_BUF_SLOTS: {
            // valid, pos, tok rows of the slot ring
            DevState st;
            CK(H, cudaMemcpyAsync(&st, h.st, sizeof(DevState), cudaMemcpyDeviceToHost, H->s_main));
            CK(H, cudaStreamSynchronize(H->s_main));
            std::vector<int> v(3 * (h.n + 1));
            for (int i = 0; i <= h.n; ++i) {
                v[i] = st.valid[i];
                v[h.n + 1 + i] = st.pos[i];
                v[2 * (h.n + 1) + i] = st.tok[i];
            }
            const size_t sz = v.size() * sizeof(int);
            if (offset > sz || bytes > sz - offset) return fail(H, SPD_EINVAL, "range outside buffer");
            std::memcpy(dst, (const char *)v.data() + offset, bytes);
            return SPD_OK;
        }
        case SPD_BUF_STATE: src = (const char *)h.st; size = 8 * sizeof(int); break;
        case SPD_BUF_PREFILL_LOGITS: src = (const char *)h.pf_logits; size = (size_t)h.V * 4; break;
        case SPD_BUF_PDM_RESIDUAL: src = (const char *)h.Xp; size = (size_t)(h.n + 1) * h.d * 4; break;
        default: return fail(H, SPD_EINVAL, "unknown buffer");
    }
    if (offset > size || bytes > size - offset) return fail(H, SPD_EINVAL, "range outside buffer");
    CK(H, cudaMemcpyAsync(dst, src + offset, bytes, cudaMemcpyDeviceToHost, H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    return SPD_OK;
}

extern "C" int spd_kernel_timing(spd_handle *H, double *total_ms, int64_t *launches) {
    if (!H) return SPD_EINVAL;
    if (!H->timing) return fail(H, SPD_ESTATE, "timing was not enabled in spd_config");
    CK(H, cudaStreamSynchronize(H->s_main));
    if (total_ms) *total_ms = H->t_ms;
    if (launches) *launches = H->t_launches;
    return SPD_OK;
}

extern "C" int spd_reset(spd_handle *H) {
    if (!H) return SPD_EINVAL;
    CK(H, cudaStreamSynchronize(H->s_main));
    CK(H, cudaMemsetAsync(H->h.st, 0, sizeof(DevState), H->s_main));
    CK(H, cudaStreamSynchronize(H->s_main));
    H->prefilled = false;
    H->t_ms = 0.0;
    H->t_launches = 0;
    return SPD_OK;
}

extern "C" void spd_destroy(spd_handle *H) {
    if (!H) return;
    if (H->s_main) cudaStreamSynchronize(H->s_main);
    if (H->g1) cudaGraphExecDestroy(H->g1);
    if (H->gN) cudaGraphExecDestroy(H->gN);
    for (auto e : H->tev)
        if (e) cudaEventDestroy(e);
    if (H->ev_fork) cudaEventDestroy(H->ev_fork);
    if (H->ev_join) cudaEventDestroy(H->ev_join);
    if (H->ev_in) cudaEventDestroy(H->ev_in);
    if (H->ev_out) cudaEventDestroy(H->ev_out);
    if (H->s_pdm) cudaStreamDestroy(H->s_pdm);
    if (H->s_main) cudaStreamDestroy(H->s_main);
    if (H->host_pinned) cudaFreeHost(H->host_pinned);
    delete H;
}

extern "C" const char *spd_last_error(const spd_handle *H) {
    return H ? H->err.c_str() : g_create_error.c_str();
}
