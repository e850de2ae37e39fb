// Target-model kernels of one pipeline step: the grouped per-stage GEMVs and the
// batched LM head.
//
// Speculative pipeline decoding (abstract; machine review "The reading"): the target is
// cut into n stages and the n in-flight tokens advance through their own stage in the
// same step.  Round j of a step runs layer b_s + j of every occupied stage s; each
// stage multiplies its own weight matrix by its own token's vector (N = 1 GEMV), so a
// round is a grouped GEMV over n different weight blocks.  The whole round's rows
// (stages x output rows) are spread evenly over the CTAs, so a partly filled pipeline
// (after a flush) still streams its weights with the whole GPU.
//
// One CTA per SM: a producer warp streams weight tiles (8 rows x up to 4 KB of each row)
// with 1-D bulk copies (TMA) into a 4-stage shared-memory ring, signalled by mbarriers;
// 8 consumer warps stage the input vector x (RMS-normalised where the layer needs it)
// while the first tiles are already in flight; then warp q owns row q of every tile of a
// group across all its K chunks, so a row ends with one warp shuffle tree and no CTA
// barrier.  Per output row the arithmetic is fixed (each lane accumulates its 16-byte
// pieces chunk by chunk in order, then the shuffle tree), so a token's result does not
// depend on which other stages share the launch: the pipeline produces bit-identical
// hidden states to a one-token-at-a-time decode.  The gate/up round stores raw gate and
// up sums; the down round forms SiLU(gate) * up while staging its input.
#include "common.cuh"

namespace spd {

enum { EPI_QKV = 0, EPI_OPROJ = 1, EPI_GATEUP = 2, EPI_DOWN = 3, EPI_LM = 4 };

constexpr int TG_CONSUMERS = 256;               // 8 consumer warps
constexpr int TG_THREADS = TG_CONSUMERS + 32;   // + 1 producer warp
constexpr int TG_RG = 8;                        // weight rows per tile
constexpr int TG_ROWB = 4096;                   // bytes of one row's chunk in a tile
constexpr int TG_NS = 4;                        // ring stages
constexpr int TG_STAGE = TG_RG * TG_ROWB;       // 32 KB
constexpr int BAR_C = 1;                        // named barrier of the consumer warps

struct StageList {
    int m;
    int stage[MAXS], slot[MAXS], layer[MAXS];
};

// Occupied stages that have a layer at this round.
__device__ void build_stage_list(const Plan *__restrict__ P, int round, StageList &L) {
    const DevState *st = P->st;
    const int n = P->n, ns = n + 1, head = st->head;
    int m = 0;
    for (int s = 0; s < n; ++s) {
        const int slot = ring(head, s, ns);
        if (!st->valid[slot]) continue;
        const int layer = P->b[s] + round;
        if (layer >= P->b[s + 1]) continue;
        L.stage[m] = s;
        L.slot[m] = slot;
        L.layer[m] = layer;
        ++m;
    }
    L.m = m;
}

// ---- consumer-only (256-thread) staging helpers: loads batched, named barrier --------
__device__ __forceinline__ float c_block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[w] = v;
    named_sync(BAR_C, TG_CONSUMERS);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < TG_CONSUMERS / 32; ++i) s += red[i];
    named_sync(BAR_C, TG_CONSUMERS);
    return s;
}

__device__ __forceinline__ void c_stage_f4(const float *__restrict__ src, float *dst, int n) {
    const int n4 = n >> 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int b = threadIdx.x; b < n4; b += 8 * TG_CONSUMERS) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * TG_CONSUMERS;
            if (i < n4) v[u] = s4[i];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * TG_CONSUMERS;
            if (i < n4) d4[i] = v[u];
        }
    }
}

// xs[k] = silu(gu[k]) * gu[F + k] (gate and up sums of the previous kernel)
__device__ __forceinline__ void c_stage_swiglu(const float *__restrict__ gu, float *xs, int F) {
    const int n4 = F >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(gu);
    const float4 *u4 = reinterpret_cast<const float4 *>(gu + F);
    float4 *d4 = reinterpret_cast<float4 *>(xs);
    for (int b = threadIdx.x; b < n4; b += 4 * TG_CONSUMERS) {
        float4 gv[4], uv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = b + u * TG_CONSUMERS;
            if (i < n4) {
                gv[u] = g4[i];
                uv[u] = u4[i];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = b + u * TG_CONSUMERS;
            if (i < n4)
                d4[i] = make_float4(silu_f(gv[u].x) * uv[u].x, silu_f(gv[u].y) * uv[u].y, silu_f(gv[u].z) * uv[u].z,
                                    silu_f(gv[u].w) * uv[u].w);
        }
    }
}

// xs = rms(x) * g over d (x staged first, fixed-order reduction); ends with a barrier
__device__ void c_stage_norm(const float *__restrict__ x, const float *__restrict__ g, int d, float eps, float *xs,
                             float *red) {
    c_stage_f4(x, xs, d);
    named_sync(BAR_C, TG_CONSUMERS);
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += TG_CONSUMERS) ss = fmaf(xs[k], xs[k], ss);
    ss = c_block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    const int d4 = d >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    float4 *x4 = reinterpret_cast<float4 *>(xs);
    for (int b = threadIdx.x; b < d4; b += 8 * TG_CONSUMERS) {
        float4 gv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * TG_CONSUMERS;
            if (i < d4) gv[u] = g4[i];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * TG_CONSUMERS;
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
    named_sync(BAR_C, TG_CONSUMERS);
}

// Weight row pointer of tile row q of the group starting at unit g0 (nullptr: no row).
template <typename T, int EPI, bool TIED>
__device__ __forceinline__ const T *tile_row(const Plan *__restrict__ P, const LayerW &w, int g0, int q, int r1, int K) {
    if (EPI == EPI_GATEUP || (EPI == EPI_LM && !TIED)) {
        const int u = g0 + (q & 3);
        if (u >= r1) return nullptr;
        const void *base;
        if (EPI == EPI_GATEUP) base = q < 4 ? w.wg : w.wu;
        else base = q < 4 ? P->lm_head : P->pdm_lm_head;
        return reinterpret_cast<const T *>(base) + (long long)u * K;
    }
    const int r = g0 + q;
    if (r >= r1) return nullptr;
    if (EPI == EPI_LM) return reinterpret_cast<const T *>(P->lm_head) + (long long)r * K;
    if (EPI == EPI_OPROJ) return reinterpret_cast<const T *>(w.wo) + (long long)r * K;
    if (EPI == EPI_DOWN) return reinterpret_cast<const T *>(w.wd) + (long long)r * K;
    if (r < P->q_rows) return reinterpret_cast<const T *>(w.wq) + (long long)r * K;
    if (r < P->q_rows + P->kv_rows) return reinterpret_cast<const T *>(w.wk) + (long long)(r - P->q_rows) * K;
    return reinterpret_cast<const T *>(w.wv) + (long long)(r - P->q_rows - P->kv_rows) * K;
}

template <typename T, int EPI, bool TIED>
__global__ void __launch_bounds__(TG_THREADS, 1) k_gemv(const Plan *__restrict__ P, int round) {
    extern __shared__ __align__(128) unsigned char tg_smem[];
    constexpr int NRHS = EPI == EPI_LM ? 2 : 1;
    constexpr int VEC = WTraits<T>::VEC;
    // units per tile group: rows, or (gate, up) / (head 0, head 1) row pairs
    constexpr int GR = (EPI == EPI_GATEUP || (EPI == EPI_LM && !TIED)) ? TG_RG / 2 : TG_RG;
    unsigned char *stages = tg_smem;
    float *xs = reinterpret_cast<float *>(tg_smem + TG_NS * TG_STAGE);
    __shared__ __align__(8) uint64_t full[TG_NS], empty[TG_NS];
    __shared__ StageList SL;
    __shared__ float cred[TG_CONSUMERS / 32];
    __shared__ int s_done, s_rows[2], s_last;
    __shared__ float s_bv[2][TG_CONSUMERS / 32];
    __shared__ int s_bi[2][TG_CONSUMERS / 32];
    const DevState *st = P->st;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        s_done = st->done;
        if (EPI == EPI_LM) {
            const int n = P->n, ns = n + 1, head = st->head;
            s_rows[0] = st->valid[ring(head, n - 1, ns)] ? ring(head, n - 1, ns) : -1;   // exit slot
            int R = st->pending ? 1 : 0;
            for (int s = 0; s < n; ++s) R += st->valid[ring(head, s, ns)] ? 1 : 0;
            s_rows[1] = R - 1;                                                          // newest draft row
            SL.m = 1;
            SL.stage[0] = SL.slot[0] = SL.layer[0] = 0;
        } else {
            build_stage_list(P, round, SL);
        }
        for (int i = 0; i < TG_NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], TG_CONSUMERS / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (s_done || SL.m == 0) return;

    const int d = P->d;
    const int N = EPI == EPI_QKV ? P->qkv_rows : EPI == EPI_GATEUP ? P->F : EPI == EPI_LM ? P->V : d;
    const int K = (EPI == EPI_QKV || EPI == EPI_GATEUP || EPI == EPI_LM) ? d : (EPI == EPI_OPROJ ? P->q_rows : P->F);
    const int nch = (int)(((long long)K * sizeof(T) + TG_ROWB - 1) / TG_ROWB);
    const int KC = ((K + nch - 1) / nch + VEC - 1) / VEC * VEC;
    const long long total = (long long)SL.m * N;
    const long long lo = total * blockIdx.x / gridDim.x;
    const long long hi = total * (blockIdx.x + 1) / gridDim.x;

    if (warp == TG_CONSUMERS / 32) {
        // ------------------------------ producer --------------------------------------
        if (lane == 0) {
            uint32_t tile = 0;
            for (long long r = lo; r < hi;) {
                const int i = (int)(r / N);
                const int r0 = (int)(r - (long long)i * N);
                const int r1 = (int)min((long long)N, hi - (long long)i * N);
                const LayerW &w = P->tl[SL.layer[i]];
                for (int g0 = r0; g0 < r1; g0 += GR) {
                    const T *rp[TG_RG];
                    int nrows = 0;
#pragma unroll
                    for (int q = 0; q < TG_RG; ++q) {
                        rp[q] = tile_row<T, EPI, TIED>(P, w, g0, q, r1, K);
                        nrows += rp[q] != nullptr;
                    }
                    for (int c = 0; c < nch; ++c) {
                        const int kc0 = c * KC, len = min(KC, K - kc0);
                        const int sidx = tile % TG_NS;
                        const uint32_t u = tile / TG_NS;
                        if (!mbar_wait(&empty[sidx], (u & 1) ^ 1)) P->st->error = ERR_TIMEOUT;
                        const uint32_t bytes = (uint32_t)len * sizeof(T);
                        mbar_expect_tx(&full[sidx], bytes * nrows);
#pragma unroll
                        for (int q = 0; q < TG_RG; ++q)
                            if (rp[q]) bulk_g2s(stages + sidx * TG_STAGE + q * TG_ROWB, rp[q] + kc0, bytes, &full[sidx]);
                        ++tile;
                    }
                }
                r = (long long)(i + 1) * N;
            }
        }
        return;
    }

    // ------------------------------ consumers -----------------------------------------
    const int tid = threadIdx.x;
    float bv[2] = {-INFINITY, -INFINITY};
    int bi[2] = {0x7fffffff, 0x7fffffff};
    const int newslot = ring(st->head + 1, 0, P->n + 1);
    float *dl = (EPI == EPI_LM && P->temperature > 0.f) ? P->dlogits + (long long)newslot * P->V : nullptr;
    uint32_t tile = 0;
    for (long long r = lo; r < hi;) {
        const int i = (int)(r / N);
        const int r0 = (int)(r - (long long)i * N);
        const int r1 = (int)min((long long)N, hi - (long long)i * N);
        const int s = SL.stage[i], slot = SL.slot[i], layer = SL.layer[i];
        const LayerW &w = P->tl[layer];
        // ---- stage x for this problem (overlaps the producer's first tiles); every warp
        // must be done with the previous problem's x first
        if (r != lo) named_sync(BAR_C, TG_CONSUMERS);
        if (EPI == EPI_QKV) c_stage_norm(P->X + (long long)slot * d, w.g1, d, P->eps, xs, cred);
        else if (EPI == EPI_GATEUP) c_stage_norm(P->X + (long long)slot * d, w.g2, d, P->eps, xs, cred);
        else if (EPI == EPI_OPROJ) {
            c_stage_f4(P->ATT + (long long)s * P->q_rows, xs, K);
            named_sync(BAR_C, TG_CONSUMERS);
        } else if (EPI == EPI_DOWN) {
            c_stage_swiglu(P->U + (long long)s * 2 * P->F, xs, K);
            named_sync(BAR_C, TG_CONSUMERS);
        } else {
            if (s_rows[0] >= 0) c_stage_norm(P->X + (long long)s_rows[0] * d, P->gf, d, P->eps, xs, cred);
            else {
                for (int k = tid; k < d; k += TG_CONSUMERS) xs[k] = 0.f;
                named_sync(BAR_C, TG_CONSUMERS);
            }
            if (P->Ls > 0) c_stage_norm(P->Xp + (long long)s_rows[1] * d, P->pdm_gf, d, P->eps, xs + d, cred);
            else {
                for (int k = tid; k < d; k += TG_CONSUMERS) xs[d + k] = 0.f;
                named_sync(BAR_C, TG_CONSUMERS);
            }
        }
        for (int g0 = r0; g0 < r1; g0 += GR) {
            // warp q owns tile row q for all chunks of this group
            const int q = warp;
            const int unit = (GR == TG_RG) ? g0 + q : g0 + (q & 3);
            const bool rv = unit < r1;
            float acc0 = 0.f, acc1 = 0.f;
            for (int c = 0; c < nch; ++c) {
                const int kc0 = c * KC, len = min(KC, K - kc0);
                const int sidx = tile % TG_NS;
                const uint32_t u = tile / TG_NS;
                if (!mbar_wait(&full[sidx], u & 1)) P->st->error = ERR_TIMEOUT;
                if (rv) {
                    const unsigned char *tb = stages + sidx * TG_STAGE + q * TG_ROWB;
                    const int nvec = len / VEC;
                    const float *xk = xs + kc0;
                    const float *xk1 = (EPI == EPI_LM) ? (TIED ? xs + d + kc0 : (q < 4 ? xs + kc0 : xs + d + kc0)) : xk;
                    for (int v = lane; v < nvec; v += 32) {
                        const uint4 wv = *reinterpret_cast<const uint4 *>(tb + v * 16);
                        if (EPI == EPI_LM && TIED) {
                            acc0 = dot16(wv, xk + v * VEC, acc0, T());
                            acc1 = dot16(wv, xk1 + v * VEC, acc1, T());
                        } else {
                            acc0 = dot16(wv, xk1 + v * VEC, acc0, T());
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[sidx]);
                ++tile;
            }
            acc0 = warp_sum(acc0);
            if (EPI == EPI_LM && TIED) acc1 = warp_sum(acc1);
            if (lane == 0 && rv) {
                if (EPI == EPI_QKV) {
                    P->QKV[(long long)s * P->qkv_rows + unit] = acc0;
                } else if (EPI == EPI_OPROJ) {
                    P->X[(long long)slot * d + unit] += acc0;
                } else if (EPI == EPI_GATEUP) {
                    // raw gate (rows 0..3) and up (rows 4..7) sums; SiLU(gate) * up is formed when
                    // the down projection stages its input
                    P->U[(long long)s * 2 * P->F + (q < 4 ? 0 : P->F) + unit] = acc0;
                } else if (EPI == EPI_DOWN) {
                    float *xp = P->X + (long long)slot * d + unit;
                    const float xn = *xp + acc0;
                    *xp = xn;
                    const int a = P->aidx[layer + 1];
                    if (a >= 0) P->ANCH[((long long)slot * P->nB + a) * d + unit] = xn;
                } else {
                    // logits: tied -> both rows of this vocab id; untied -> row (q >= 4) only
                    const int h0 = TIED ? 0 : (q < 4 ? 0 : 1);
                    for (int h = h0; h < (TIED ? 2 : h0 + 1); ++h) {
                        const float z = h == h0 ? acc0 : acc1;
                        P->logits[(long long)h * P->V + unit] = z;
                        if (h == 1 && dl) dl[unit] = z;
                        if (z > bv[h] || (z == bv[h] && unit < bi[h])) {
                            bv[h] = z;
                            bi[h] = unit;
                        }
                    }
                }
            }
        }
        r = (long long)(i + 1) * N;
    }
    if (EPI != EPI_LM) return;

    // ---- LM head: CTA argmax (lowest id on ties; candidates in lane 0 of every warp),
    // then the last CTA merges the CTA results in CTA order
    if (lane == 0) {
        s_bv[0][warp] = bv[0];
        s_bi[0][warp] = bi[0];
        s_bv[1][warp] = bv[1];
        s_bi[1][warp] = bi[1];
    }
    named_sync(BAR_C, TG_CONSUMERS);
    if (tid < 2) {
        float cv = -INFINITY;
        int ci = 0x7fffffff;
        for (int w2 = 0; w2 < TG_CONSUMERS / 32; ++w2)
            if (s_bv[tid][w2] > cv || (s_bv[tid][w2] == cv && s_bi[tid][w2] < ci)) {
                cv = s_bv[tid][w2];
                ci = s_bi[tid][w2];
            }
        P->lm_part[blockIdx.x * 4 + tid * 2] = cv;
        P->lm_part[blockIdx.x * 4 + tid * 2 + 1] = __int_as_float(ci);
    }
    __threadfence();
    named_sync(BAR_C, TG_CONSUMERS);
    if (tid == 0) s_last = atomicAdd(P->lm_cnt, 1) == (int)gridDim.x - 1;
    named_sync(BAR_C, TG_CONSUMERS);
    if (!s_last) return;
    __threadfence();
    for (int row = 0; row < 2; ++row) {
        float cv = -INFINITY;
        int ci = 0x7fffffff;
        for (int c = tid; c < (int)gridDim.x; c += TG_CONSUMERS) {
            const float v = __ldcg(P->lm_part + c * 4 + row * 2);
            const int id = __float_as_int(__ldcg(P->lm_part + c * 4 + row * 2 + 1));
            if (v > cv || (v == cv && id < ci)) {
                cv = v;
                ci = id;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, cv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, ci, o);
            if (ov > cv || (ov == cv && oi < ci)) {
                cv = ov;
                ci = oi;
            }
        }
        if (lane == 0) {
            s_bv[row][warp] = cv;
            s_bi[row][warp] = ci;
        }
    }
    named_sync(BAR_C, TG_CONSUMERS);
    if (tid < 2) {
        const int row = tid;
        float cv = -INFINITY;
        int ci = 0x7fffffff;
        for (int w2 = 0; w2 < TG_CONSUMERS / 32; ++w2) {
            const float v = s_bv[row][w2];
            const int id = s_bi[row][w2];
            if (v > cv || (v == cv && id < ci)) {
                cv = v;
                ci = id;
            }
        }
        P->st->top[row] = ci;
        P->st->topval[row] = cv;
    }
    if (tid == 0) *P->lm_cnt = 0;
}

// ---------------------------------------------------------------------------------
static int x_bytes(const Plan &h, int epi) {
    const int K = (epi == EPI_QKV || epi == EPI_GATEUP) ? h.d
                  : epi == EPI_OPROJ                  ? h.q_rows
                  : epi == EPI_DOWN                   ? h.F
                                                      : 2 * h.d;
    return K * (int)sizeof(float);
}
static int smem_for(const Plan &h, int epi) { return TG_NS * TG_STAGE + x_bytes(h, epi); }

template <typename T, int EPI>
static void launch_epi(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    k_gemv<T, EPI, true><<<grid, TG_THREADS, smem_for(h, EPI), s>>>(P, round);
}

template <typename T>
void launch_target_qkv(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    launch_epi<T, EPI_QKV>(P, h, round, grid, s);
}
template <typename T>
void launch_target_oproj(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    launch_epi<T, EPI_OPROJ>(P, h, round, grid, s);
}
template <typename T>
void launch_target_gateup(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    launch_epi<T, EPI_GATEUP>(P, h, round, grid, s);
}
template <typename T>
void launch_target_down(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    launch_epi<T, EPI_DOWN>(P, h, round, grid, s);
}
template <typename T>
void launch_lm_head(const Plan *P, const Plan &h, int grid, cudaStream_t s) {
    if (h.pdm_lm_head == h.lm_head)
        k_gemv<T, EPI_LM, true><<<grid, TG_THREADS, smem_for(h, EPI_LM), s>>>(P, 0);
    else
        k_gemv<T, EPI_LM, false><<<grid, TG_THREADS, smem_for(h, EPI_LM), s>>>(P, 0);
}

int gemv_smem_bytes(const Plan &h) {
    int m = 0;
    for (int e = 0; e <= EPI_LM; ++e) m = smem_for(h, e) > m ? smem_for(h, e) : m;
    return m;
}
int target_blocks_per_sm(int, int) { return 1; }
int lm_blocks_per_sm(int, int, bool) { return 1; }

template <typename T>
static void set_attr_t(int smem) {
    cudaFuncSetAttribute(k_gemv<T, EPI_QKV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<T, EPI_OPROJ, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<T, EPI_GATEUP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<T, EPI_DOWN, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<T, EPI_LM, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<T, EPI_LM, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}
void set_target_attributes(int smem) {
    set_attr_t<float>(smem);
    set_attr_t<__nv_bfloat16>(smem);
}

#define INST(T)                                                                                   \
    template void launch_target_qkv<T>(const Plan *, const Plan &, int, int, cudaStream_t);       \
    template void launch_target_oproj<T>(const Plan *, const Plan &, int, int, cudaStream_t);     \
    template void launch_target_gateup<T>(const Plan *, const Plan &, int, int, cudaStream_t);    \
    template void launch_target_down<T>(const Plan *, const Plan &, int, int, cudaStream_t);      \
    template void launch_lm_head<T>(const Plan *, const Plan &, int, cudaStream_t);
INST(float)
INST(__nv_bfloat16)
#undef INST

}  // namespace spd
