// Shared device-side definitions of the speculative-pipeline-decoding library.
//
// Layout of the run state in HBM (all carved out of the caller's workspace):
//   slot ring     n+1 slots; stage s of the current step lives in slot (head - s) mod (n+1),
//                 the token that left the last stage in the previous step ("exited row",
//                 read once more by the draft module) in slot (head - n) mod (n+1).
//   X   fp32 [n+1][d]            residual stream per slot
//   ANCH fp32 [n+1][nB][d]       anchor states per slot (depth a = after a layers, 0 = embedding)
//   QKV fp32 [n][(Hq+2Hkv) hd]   raw q,k,v of each stage (RoPE is applied by the attention kernel)
//   att_part fp32 [stage][Hq][chunk][hd+4]  attention chunk partials (merged by the O projection)
//   U   fp32 [n][2F]             raw gate and up sums of each stage (SiLU(gate)*up formed by the down GEMV)
//   K/V cache per target layer   fp32 [max_seq][Hkv][hd]; valid length per layer in DevState
//   draft module buffers         Xp [n+1][d], QKVp/ATTp/GUp per row, its own K/V cache
//   logits fp32 [2][V]           row 0 = target prediction of the exiting token, row 1 = draft
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spd.h"

namespace spd {

constexpr int MAXS = 32;                 // ring slots (n + 1 <= 32)
constexpr int MAXL = SPD_MAX_LAYERS;
constexpr int MAXPL = SPD_MAX_PDM_LAYERS;
constexpr int MAXB = SPD_MAX_ANCHORS;
constexpr int ATT_CHUNK = 128;           // positions per attention split (fixed: results independent of grouping)
// floats per attention partial row (one head, one chunk): o[hd], max, sum, 2 pad (16-byte rows)
__host__ __device__ constexpr int att_part_pitch(int hd) { return hd + 4; }
constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int MAX_R = MAXS;              // draft-module rows per step (n+1)

// device error codes (DevState::error)
constexpr int ERR_FORCED_REF = 1;
constexpr int ERR_TRACE_FULL = 2;
constexpr int ERR_SEQ_FULL = 3;
constexpr int ERR_ROWS = 4;
constexpr int ERR_TOKEN = 5;
constexpr int ERR_TIMEOUT = 6;   // a bounded mbarrier wait gave up

struct LayerW {
    const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
    const float *g1, *g2;
};

struct DevState {
    int head, t, N, done, pending, error, pdm_len, prompt_len;   // first 8: SPD_BUF_STATE
    int valid[MAXS], pos[MAXS], tok[MAXS];
    int len[MAXL];
    // argmax results of the last LM-head pass (row 0 target, row 1 draft)
    int top[2];
    float topval[2];
    // draft distribution normalisers per slot (T > 0): max and sum of exp(z/T - max)
    float dmax[MAXS], dsum[MAXS];
    // T > 0, tensor-core LM head: the draft token it sampled, and both rows' softmax
    // normalisers (max of z/T, sum of exp(z/T - max)), row 0 target, row 1 draft
    int samp, pad_[3];
    float lmM[2], lmS[2];
    long long accepts, rejects, run_cur, run_sum, run_count;
    double weight_bytes;
};

// Constant description of one handle: shapes, stage plan, weight and buffer pointers.
struct Plan {
    int L, d, Hq, Hkv, hd, F, V, n, nB, Ls, max_seq, max_new, max_steps, dtype;
    int qkv_rows, q_rows, kv_rows;
    int J;                         // rounds per step = longest stage
    int b[MAXS + 1];               // stage bounds
    int spec_out;                  // 1: the draft module runs after the step on its output states
    int anchors[MAXB];
    signed char aidx[MAXL + 1];    // anchor index of depth a, or -1
    float eps, scale, temperature;
    unsigned seed_lo, seed_hi;
    int forced;
    unsigned forced_thr;           // coin: u24 < forced_thr keeps forced_ref
    const int *forced_ref;
    int forced_ref_len;
    // weights
    const void *embed, *lm_head, *pdm_lm_head, *proj;
    const float *gf, *pdm_gf;
    LayerW tl[MAXL];
    LayerW pl[MAXPL];
    // workspace
    float *X, *QKV, *U, *ANCH;   // U: [n][2F] gate | up
    void *kc, *vc, *pkc, *pvc;
    long long kv_stride;           // elements per layer cache
    float2 *rope;                  // [max_seq][hd/2] (cos, sin)
    float *att_part, *patt_part;   // [MAXS][Hq][max_chunks][hd + 4] (target per stage / draft module per row)
    int *att_cnt, *patt_cnt;       // [MAXS][Hkv]
    int att_max_chunks;
    long long layer_bytes;         // weight bytes of one target layer
    long long pdm_bytes;           // draft module per step (projection + layers)
    long long lm_bytes;            // LM head per step
    float *Xp, *QKVp, *ATTp, *GUp;  // draft module rows: residual, q|k|v, attention, SiLU(gate)*up
    float *ssp;                    // [MAXS][d / 8] sums of squares of 8-row groups of the Xp rows
    // bf16 weights: the draft GEMMs' inputs as bf16 rows, copied into shared memory whole; each
    // buffer holds the rows' hi parts bf16(x), then (same layout, right after) their lo parts
    // bf16(x - hi)
    __nv_bfloat16 *Xb;             // 2 x [n+1][d] Xp * g of the next normalisation (1/rms applied after the GEMM)
    __nv_bfloat16 *ATTb;           // 2 x [n+1][Hq hd] attention output
    __nv_bfloat16 *GUb;            // 2 x [n+1][F] SiLU(gate) * up
    __nv_bfloat16 *ANCHb;          // 2 x [n+1][nB][d] the anchor states (the draft projection's input)
    __nv_bfloat16 *Xlm;            // [4][d] LM head rows: x * g_final of the exiting token and of the draft's newest row
                                   // (rows 0, 1: bf16 of the value; rows 2, 3: bf16 of what rows 0, 1 left out)
    float *pdm_part;               // draft GEMM K-slab partials [slab][n+1][N]
    int *pdm_cnt;                  // draft GEMM row-block arrival counters (zero between launches)
    int pdm_kx[6], pdm_ns[6];      // draft-style GEMMs (proj, qkv, o, gate/up, down, LM head): K slab width, slabs
    int pdm_MT;                    // 16-row mma tiles of the draft rows (1: n+1 <= 16, else 2)
    int pdl;                       // step kernels launched with programmatic dependent launch
    long long wait_cycles;         // bound of the grouped GEMV's mbarrier waits (SM cycles)
    int test_withhold;             // test hook: 1 = the first gate/up launch's CTA 0 never loads its last tile
    float *logits;                 // [2][V]
    float *dlogits;                // [n+1][V] draft logits per slot (T > 0)
    float *lm_part;                // [grid][2] (val, idx as float bits)
    float *lm_stat;                // [grid][2] (max of z/T, sum of exp(z/T - max)) per LM-head CTA and row (T > 0)
    int lm_stats;                  // 1: the tensor-core LM head leaves the T > 0 statistics and the draft sample
    int *lm_cnt;
    DevState *st;
    spd_trace_rec *trace;
    int *trace_len;                // [max_steps][L]
    int *out_tokens;               // [max_new]
    // prefill scratch
    int pf_rows;                   // rows per prefill chunk
    float *pf_H, *pf_XN, *pf_QKV, *pf_ATT, *pf_GU, *pf_ANCH, *pf_Hp;
    float *pf_logits;              // [V]
    __nv_bfloat16 *pf_A2;          // bf16 weights: the tensor-core GEMMs' input rows as two bf16 parts,
                                   // hi [pf_rows][K] then lo [pf_rows][K], K the consuming GEMM's width
    Plan *self;                    // device address of this plan
};

// ---------------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (TMA) helpers.  Every wait is bounded in time: on timeout the
// caller records an error flag and carries on (no trap, no endless spin).
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
constexpr long long WAIT_LIMIT_CYCLES = 4000000000ll;   // ~2 s of SM clock: far beyond any legitimate wait
// Wait for the completion of the phase with this parity; false after `limit` cycles.
// The bound uses the SM's own cycle counter, which is cheap to read inside the spin.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit = WAIT_LIMIT_CYCLES) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}
// 1-D bulk copy global -> this CTA's shared memory; completion counted in bytes on bar.
// src, dst and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// Orders this thread's generic-proxy memory accesses before its later bulk copies.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
// Asynchronous 16-byte global -> shared copy (no register staging); wait_all waits for all
// of the thread's outstanding copies.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Programmatic dependent launch.  Step kernels are launched so that the next kernel of the
// stream may start while this one drains: pdl_wait() blocks until the preceding kernel has
// completed and its writes are visible (a no-op when it was launched without the attribute);
// pdl_trigger() lets the following kernel start once every CTA of this one has triggered or
// exited.  Each kernel triggers only after its own wait, so when a kernel starts, every
// kernel before its predecessor has completed: before its wait it may read weights and the
// step-stable slot state, nothing its predecessor writes, and it writes nothing global.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Barrier among the first `threads` threads of the CTA (id 0 is __syncthreads').
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------------
// element access
template <typename T> struct WTraits;
template <> struct WTraits<float> {
    static constexpr int VEC = 4;   // elements per 16-byte load
    __device__ static __forceinline__ float get(const float *p, long long i) { return p[i]; }
    __device__ static __forceinline__ float store(float v) { return v; }
};
template <> struct WTraits<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ static __forceinline__ float get(const __nv_bfloat16 *p, long long i) { return __bfloat162float(p[i]); }
    __device__ static __forceinline__ __nv_bfloat16 store(float v) { return __float2bfloat16_rn(v); }
};
// fp16: a K/V operand type of the stand-alone attention call.  Values beyond the fp16 range
// saturate at +-65504 instead of becoming infinite.
constexpr float F16_MAX = 65504.f;
template <> struct WTraits<__half> {
    static constexpr int VEC = 8;
    __device__ static __forceinline__ float get(const __half *p, long long i) { return __half2float(p[i]); }
    __device__ static __forceinline__ __half store(float v) { return __float2half_rn(fminf(fmaxf(v, -F16_MAX), F16_MAX)); }
};

// Element type of the K/V caches for weights of type T: fp32 for every model.  Every later
// token attends over every cached row, so the cache's rounding reaches all logits: with fp16
// rows (bf16 rows are 8x coarser) an 8B-shaped random-init model's logits moved by 2-3e-2 of
// their scale, K and V contributing about equally; fp32 rows leave the cache exact to fp32.
template <typename T> using KvT = float;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float h_lo(uint32_t u) { return __half2float(__ushort_as_half((unsigned short)(u & 0xffffu))); }
__device__ __forceinline__ float h_hi(uint32_t u) { return __half2float(__ushort_as_half((unsigned short)(u >> 16))); }

// Dot product of one 16-byte weight vector with the matching x values (fixed order).
__device__ __forceinline__ float dot16(const uint4 &w, const float *x, float acc, __nv_bfloat16) {
    const float4 x0 = *reinterpret_cast<const float4 *>(x);
    const float4 x1 = *reinterpret_cast<const float4 *>(x + 4);
    acc = fmaf(bf_lo(w.x), x0.x, acc);
    acc = fmaf(bf_hi(w.x), x0.y, acc);
    acc = fmaf(bf_lo(w.y), x0.z, acc);
    acc = fmaf(bf_hi(w.y), x0.w, acc);
    acc = fmaf(bf_lo(w.z), x1.x, acc);
    acc = fmaf(bf_hi(w.z), x1.y, acc);
    acc = fmaf(bf_lo(w.w), x1.z, acc);
    acc = fmaf(bf_hi(w.w), x1.w, acc);
    return acc;
}
__device__ __forceinline__ float dot16(const uint4 &w, const float *x, float acc, float) {
    const float4 x0 = *reinterpret_cast<const float4 *>(x);
    acc = fmaf(__uint_as_float(w.x), x0.x, acc);
    acc = fmaf(__uint_as_float(w.y), x0.y, acc);
    acc = fmaf(__uint_as_float(w.z), x0.z, acc);
    acc = fmaf(__uint_as_float(w.w), x0.w, acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum with a fixed reduction tree (result broadcast to all threads).
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    if (w == 0) {
        s = lane < nw ? red[lane] : 0.f;
        s = warp_sum(s);
        if (lane == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}
__device__ __forceinline__ float block_max(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = -INFINITY;
    if (w == 0) {
        s = lane < nw ? red[lane] : -INFINITY;
        s = warp_max(s);
        if (lane == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}

// Copy n floats (n % 4 == 0, both 16-byte aligned) from global to shared memory with up
// to 8 16-byte loads per thread in flight before any store.  Kept out of line so that its
// staging registers do not count against the caller's main loop.
static __device__ __noinline__ void stage_f4(const float *__restrict__ src, float *dst, int n) {
    const int n4 = n >> 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int b = threadIdx.x; b < n4; b += 8 * blockDim.x) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * blockDim.x;
            if (i < n4) v[u] = s4[i];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * blockDim.x;
            if (i < n4) d4[i] = v[u];
        }
    }
}

// x staging of a normalised input: xs = rms(x) * g.  x is staged first, the statistics
// come from shared memory with a fixed-order block reduction.  Ends with __syncthreads.
static __device__ __noinline__ void stage_norm(const float *__restrict__ x, const float *__restrict__ g, int d, float eps,
                                        float *xs, float *red) {
    stage_f4(x, xs, d);
    __syncthreads();
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float v = xs[k];
        ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    const int d4 = d >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    float4 *x4 = reinterpret_cast<float4 *>(xs);
    for (int b = threadIdx.x; b < d4; b += 8 * blockDim.x) {
        float4 gv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * blockDim.x;
            if (i < d4) gv[u] = g4[i];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * blockDim.x;
            if (i < d4) {
                float4 v = x4[i];
                v.x = (v.x * inv) * gv[u].x;
                v.y = (v.y * inv) * gv[u].y;
                v.z = (v.z * inv) * gv[u].z;
                v.w = (v.w * inv) * gv[u].w;
                x4[i] = v;
            }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int ring(int head, int s, int nslots) {
    int r = (head - s) % nslots;
    return r < 0 ? r + nslots : r;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Philox4x32-10 (Salmon et al., SC'11): two 32x32->64-bit multiplies per round,
// Weyl-sequence key schedule, ten rounds.  Counter (t, purpose, 0, 0), key (lo, hi).
__device__ __forceinline__ uint32_t philox_word0(uint32_t t, uint32_t purpose, uint32_t klo, uint32_t khi) {
    uint32_t c0 = t, c1 = purpose, c2 = 0u, c3 = 0u;
    uint32_t k0 = klo, k1 = khi;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

// Rows of the draft module in the current step: the token that left the pipeline in
// the previous step (all anchors, cached permanently from now on), then the in-flight
// tokens oldest first; consecutive positions pos0, pos0+1, ...
struct PdmRows {
    int R, pos0;
    int slot[MAXS], depth[MAXS], pos[MAXS];
};

// Occupied stages that have a layer at this round, in stage order.
struct StageList {
    int m;
    int stage[MAXS], slot[MAXS], layer[MAXS], pos[MAXS];
};

// Both are built by one full warp (lane s looks at stage s, so the slot-ring reads of all
// stages are in flight together).  Only the calling warp sees the result until the CTA
// synchronises.
__device__ __forceinline__ void warp_stage_list(const Plan *__restrict__ P, int round, StageList &L, int *done) {
    const int lane = threadIdx.x & 31;
    const DevState *st = P->st;
    const int n = P->n, head = st->head;
    bool ok = false;
    int slot = 0, layer = 0, pos = 0;
    if (lane < n) {
        slot = ring(head, lane, n + 1);
        const int v = st->valid[slot];
        const int b0 = P->b[lane], b1 = P->b[lane + 1];
        pos = st->pos[slot];
        layer = b0 + round;
        ok = v && layer < b1;
    }
    const unsigned mask = __ballot_sync(0xffffffffu, ok);
    if (ok) {
        const int i = __popc(mask & ((1u << lane) - 1u));
        L.stage[i] = lane;
        L.slot[i] = slot;
        L.layer[i] = layer;
        L.pos[i] = pos;
    }
    if (lane == 0) {
        L.m = __popc(mask);
        if (done) *done = st->done;
    }
    __syncwarp();
}

// The draft module has a full-depth row for the token that left the pipeline in the
// previous step only under the input-state schedule; under the output-state schedule that
// token was at full depth in its own step already.
__device__ __forceinline__ int pdm_pending(const Plan *__restrict__ P, const DevState *st) {
    return P->spec_out ? 0 : st->pending;
}

// Input-state schedule: stage s's row at its input depth b_s; output-state schedule (the
// module runs after the step's target layers): at its output depth b_{s+1}.
__device__ __forceinline__ void warp_pdm_rows(const Plan *__restrict__ P, PdmRows &pr, int *done) {
    const int lane = threadIdx.x & 31;
    const DevState *st = P->st;
    const int n = P->n, head = st->head, pending = pdm_pending(P, st);
    bool v = false;
    int slot = 0, pos = 0, depth = 0;
    if (lane < n) {
        slot = ring(head, lane, n + 1);
        v = st->valid[slot] != 0;
        pos = st->pos[slot];
        depth = P->b[lane + P->spec_out];
    } else if (lane == n && pending) {
        slot = ring(head, n, n + 1);
        pos = st->pos[slot];
        depth = P->L;
    }
    const unsigned mask = __ballot_sync(0xffffffffu, v);
    if (v) {
        // rows: exited token first, then stages from the deepest (oldest) to stage 0
        const int i = (pending ? 1 : 0) + __popc(lane == 31 ? 0u : (mask >> (lane + 1)));
        pr.slot[i] = slot;
        pr.depth[i] = depth;
        pr.pos[i] = pos;
    } else if (lane == n && pending) {
        pr.slot[0] = slot;
        pr.depth[0] = depth;
        pr.pos[0] = pos;
    }
    __syncwarp();
    if (lane == 0) {
        pr.R = (pending ? 1 : 0) + __popc(mask);
        pr.pos0 = pr.R > 0 ? pr.pos[0] : 0;
        if (done) *done = st->done;
    }
    __syncwarp();
}

// Launch with (pdl = true) or without the programmatic-serialisation attribute.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                   Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------------
// launch helpers (defined in the kernel translation units)
template <typename T> void launch_target_round(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s);
template <typename T> void launch_target_qkv(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s);
template <typename T> void launch_target_attn(const Plan *P, const Plan &h, int round, cudaStream_t s);
template <typename T> void launch_target_oproj(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s);
template <typename T> void launch_target_gateup(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s);
template <typename T> void launch_target_down(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s);
template <typename T> void launch_lm_head(const Plan *P, const Plan &h, int grid, cudaStream_t s);
template <typename T> void launch_pdm_step(const Plan *P, const Plan &h, int grid, cudaStream_t s);
template <typename T> void launch_pdm_attn(const Plan *P, const Plan &h, int layer, cudaStream_t s);
void pdm_plan(int d, int F, int q_rows, int nB, int n, int dtype, int kx[6], int ns[6], int *MT);
template <typename T> void launch_pdm_lm(const Plan *P, const Plan &h, int grid, cudaStream_t s);
bool lm_on_tensor_cores(const Plan &h);   // the LM head runs as a tensor-core GEMM (launch_pdm_lm)
void set_pdm_attributes();
void set_target_attributes(int smem);
void set_prefill_attributes();
void set_attn_attributes();
int attn_smem_bytes(int dtype, int hd, int G);
template <typename T> void launch_verify(const Plan *P, const Plan &h, cudaStream_t s);
// returns nonzero when a tensor map could not be encoded (nothing further was launched)
template <typename T> int launch_prefill(const Plan *P, const Plan &h, const int *prompt, int prompt_len, int num_sms,
                                          cudaStream_t s);
template <typename T> void launch_prefill_finalize(const Plan *P, int prompt_len, cudaStream_t s);
void launch_rope_table(const Plan &h, float theta, cudaStream_t s);
int gemv_smem_bytes(const Plan &h);
int target_blocks_per_sm(int dtype, int smem);
int lm_blocks_per_sm(int dtype, int smem, bool tied);
void set_kernel_attributes(int dtype, int gemv_smem);

}  // namespace spd
