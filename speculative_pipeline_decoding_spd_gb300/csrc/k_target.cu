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
// One CTA per SM: a producer warp streams weight tiles (8 rows x up to 6 KB of each row)
// with 1-D bulk copies (TMA) into a shared-memory ring of as many stages as fit beside x
// (5 x 40 KB for the 4B shape's QKV and gate/up), signalled by mbarriers;
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
constexpr int TG_ROWB = 6144;                   // at most this many bytes of a row per tile chunk
constexpr int TG_MAXNS = 8;                     // ring stages (the ring fills what x leaves free)
constexpr int TG_SMEM = 210 * 1024;             // dynamic shared memory: ring + x
constexpr int BAR_C = 1;                        // named barrier of the consumer warps

// ---- consumer-only (256-thread) staging helpers: loads batched, named barrier --------
// For bf16 weights x is kept in shared memory as two planes, element 8v+j at
// xp(8v+j) = (j < 4 ? 0 : plane) + 4v + (j & 3), so the 16-byte x reads of a warp (lane v)
// are contiguous per plane and hit distinct banks.
template <typename T> __device__ __forceinline__ int xp(int k, int plane);
template <> __device__ __forceinline__ int xp<float>(int k, int) { return k; }
template <> __device__ __forceinline__ int xp<__nv_bfloat16>(int k, int plane) {
    return ((k & 4) ? plane : 0) + ((k >> 3) << 2) + (k & 3);
}
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

template <typename T>
__device__ __noinline__ void c_stage_f4(const float *__restrict__ src, float *dst, int n) {
    const int n4 = n >> 2, plane = n >> 1;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
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
            if (i < n4) *reinterpret_cast<float4 *>(dst + xp<T>(4 * i, plane)) = v[u];
        }
    }
}

// xs[k] = silu(gu[k]) * gu[F + k] (gate and up sums of the previous kernel)
template <typename T>
__device__ __noinline__ void c_stage_swiglu(const float *__restrict__ gu, float *xs, int F) {
    const int n4 = F >> 2, plane = F >> 1;
    const float4 *g4 = reinterpret_cast<const float4 *>(gu);
    const float4 *u4 = reinterpret_cast<const float4 *>(gu + F);
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
                *reinterpret_cast<float4 *>(xs + xp<T>(4 * i, plane)) =
                    make_float4(silu_f(gv[u].x) * uv[u].x, silu_f(gv[u].y) * uv[u].y, silu_f(gv[u].z) * uv[u].z,
                                silu_f(gv[u].w) * uv[u].w);
        }
    }
}

// xs = attention output of stage s: each head's chunk partials (o_c, m_c, l_c) merged in
// chunk order, x = (sum_c e^{m_c - M} o_c) / (sum_c e^{m_c - M} l_c), M = max_c m_c.
// wsm: 2 * Hq * nch floats of shared memory.  Ends with a barrier.
template <typename T>
__device__ __noinline__ void c_stage_attn(const Plan *__restrict__ P, int s, int pos, float *xs, float *wsm) {
    const int Hq = P->Hq, hd = P->hd, maxch = P->att_max_chunks, pp = att_part_pitch(hd);
    const int nch = pos / ATT_CHUNK + 1, tid = threadIdx.x;
    const float *part = P->att_part + (long long)s * Hq * maxch * pp;
    float *wl = wsm + Hq * nch;
    for (int i = tid; i < Hq * nch; i += TG_CONSUMERS) {
        const int h = i / nch, c = i - h * nch;
        const float2 ml = *reinterpret_cast<const float2 *>(part + ((long long)h * maxch + c) * pp + hd);
        wsm[i] = ml.x;
        wl[i] = ml.y;
    }
    named_sync(BAR_C, TG_CONSUMERS);
    for (int h = tid; h < Hq; h += TG_CONSUMERS) {
        float M = -INFINITY;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, wsm[h * nch + c]);
        float den = 0.f;
        for (int c = 0; c < nch; ++c) {
            const float w = expf(wsm[h * nch + c] - M);
            wsm[h * nch + c] = w;
            den = fmaf(w, wl[h * nch + c], den);
        }
        wl[h * nch] = den;
    }
    named_sync(BAR_C, TG_CONSUMERS);
    // 4-element groups, two per thread per pass with up to 8 chunks each in flight
    const int K = Hq * hd, g4 = K >> 2, q4 = hd >> 2, plane = K >> 1;
    for (int b = tid; b < g4; b += 2 * TG_CONSUMERS) {
        for (int c0 = 0; c0 < nch; c0 += 8) {
            float4 v[2][8];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = b + e * TG_CONSUMERS, h = i / q4, d4 = i - h * q4;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i < g4 && c0 + u < nch)
                        v[e][u] = *reinterpret_cast<const float4 *>(part + ((long long)h * maxch + c0 + u) * pp + 4 * d4);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = b + e * TG_CONSUMERS, h = i / q4;
                if (i >= g4) continue;
                float4 *px = reinterpret_cast<float4 *>(xs + xp<T>(4 * i, plane));
                float4 acc = c0 == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : *px;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + u < nch) {
                        const float w = wsm[h * nch + c0 + u];
                        acc.x = fmaf(w, v[e][u].x, acc.x);
                        acc.y = fmaf(w, v[e][u].y, acc.y);
                        acc.z = fmaf(w, v[e][u].z, acc.z);
                        acc.w = fmaf(w, v[e][u].w, acc.w);
                    }
                if (c0 + 8 >= nch) {
                    const float den = wl[h * nch];
                    acc = make_float4(acc.x / den, acc.y / den, acc.z / den, acc.w / den);
                }
                *px = acc;
            }
        }
    }
    named_sync(BAR_C, TG_CONSUMERS);
}

// xs = rms(x) * g over d (x staged first, fixed-order reduction); ends with a barrier
template <typename T>
__device__ __noinline__ void c_stage_norm(const float *__restrict__ x, const float *__restrict__ g, int d, float eps, float *xs,
                             float *red) {
    c_stage_f4<T>(x, xs, d);
    named_sync(BAR_C, TG_CONSUMERS);
    const int plane = d >> 1;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += TG_CONSUMERS) {
        const float v = xs[xp<T>(k, plane)];
        ss = fmaf(v, v, ss);
    }
    ss = c_block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    const int d4 = d >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
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
                float4 *px = reinterpret_cast<float4 *>(xs + xp<T>(4 * i, plane));
                float4 v = *px;
                v.x = (v.x * inv) * gv[u].x;
                v.y = (v.y * inv) * gv[u].y;
                v.z = (v.z * inv) * gv[u].z;
                v.w = (v.w * inv) * gv[u].w;
                *px = v;
            }
        }
    }
    named_sync(BAR_C, TG_CONSUMERS);
}

// One 16-byte weight vector (elements e..e+VEC-1) against x in its shared-memory layout.
template <typename T>
__device__ __forceinline__ float dot_x(const uint4 &w, const float *x, int e, int plane, float acc);
template <>
__device__ __forceinline__ float dot_x<float>(const uint4 &w, const float *x, int e, int, float acc) {
    return dot16(w, x + e, acc, 0.f);
}
template <>
__device__ __forceinline__ float dot_x<__nv_bfloat16>(const uint4 &w, const float *x, int e, int plane, float acc) {
    const float4 a = *reinterpret_cast<const float4 *>(x + (e >> 1));
    const float4 b = *reinterpret_cast<const float4 *>(x + plane + (e >> 1));
    acc = fmaf(bf_lo(w.x), a.x, acc);
    acc = fmaf(bf_hi(w.x), a.y, acc);
    acc = fmaf(bf_lo(w.y), a.z, acc);
    acc = fmaf(bf_hi(w.y), a.w, acc);
    acc = fmaf(bf_lo(w.z), b.x, acc);
    acc = fmaf(bf_hi(w.z), b.y, acc);
    acc = fmaf(bf_lo(w.w), b.z, acc);
    acc = fmaf(bf_hi(w.w), b.w, acc);
    return acc;
}

// x values that one 16-byte weight vector at element e meets, loaded once and applied to
// several weight rows (the LM head's paired tiles).
template <typename T> struct XV;
template <> struct XV<float> {
    float4 a;
    __device__ __forceinline__ void load(const float *x, int e, int) { a = *reinterpret_cast<const float4 *>(x + e); }
    __device__ __forceinline__ float dot(const uint4 &w, float acc) const {
        acc = fmaf(__uint_as_float(w.x), a.x, acc);
        acc = fmaf(__uint_as_float(w.y), a.y, acc);
        acc = fmaf(__uint_as_float(w.z), a.z, acc);
        acc = fmaf(__uint_as_float(w.w), a.w, acc);
        return acc;
    }
};
template <> struct XV<__nv_bfloat16> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *x, int e, int plane) {
        a = *reinterpret_cast<const float4 *>(x + (e >> 1));
        b = *reinterpret_cast<const float4 *>(x + plane + (e >> 1));
    }
    // same element order as dot_x<bf16>
    __device__ __forceinline__ float dot(const uint4 &w, float acc) const {
        acc = fmaf(bf_lo(w.x), a.x, acc);
        acc = fmaf(bf_hi(w.x), a.y, acc);
        acc = fmaf(bf_lo(w.y), a.z, acc);
        acc = fmaf(bf_hi(w.y), a.w, acc);
        acc = fmaf(bf_lo(w.z), b.x, acc);
        acc = fmaf(bf_hi(w.z), b.y, acc);
        acc = fmaf(bf_lo(w.w), b.z, acc);
        acc = fmaf(bf_hi(w.w), b.w, acc);
        return acc;
    }
};

// Weight rows of one problem, resolved once per segment into registers: unit u reads row
// u of region 0 below b1, row u - b1 of region 1 below b2, else row u - b2 of region 2.
// Gate/up and untied-head tiles read slot q < 4 from region 0 and q >= 4 from region 1
// for the same unit.
template <typename T>
struct SegRows {
    const T *p0, *p1, *p2;
    int b1, b2;
};

template <typename T, int EPI, bool TIED>
__device__ __forceinline__ SegRows<T> seg_rows(const Plan *__restrict__ P, const LayerW &w) {
    SegRows<T> r;
    r.b1 = r.b2 = 0x7fffffff;
    if (EPI == EPI_GATEUP) {
        r.p0 = reinterpret_cast<const T *>(w.wg);
        r.p1 = reinterpret_cast<const T *>(w.wu);
        r.p2 = nullptr;
    } else if (EPI == EPI_LM) {
        r.p0 = reinterpret_cast<const T *>(P->lm_head);
        r.p1 = reinterpret_cast<const T *>(P->pdm_lm_head);
        r.p2 = nullptr;
    } else if (EPI == EPI_OPROJ || EPI == EPI_DOWN) {
        r.p0 = reinterpret_cast<const T *>(EPI == EPI_OPROJ ? w.wo : w.wd);
        r.p1 = r.p2 = nullptr;
    } else {
        r.p0 = reinterpret_cast<const T *>(w.wq);
        r.p1 = reinterpret_cast<const T *>(w.wk);
        r.p2 = reinterpret_cast<const T *>(w.wv);
        r.b1 = P->q_rows;
        r.b2 = P->q_rows + P->kv_rows;
    }
    return r;
}

template <typename T, int EPI, bool TIED>
__device__ __forceinline__ const T *tile_row(const SegRows<T> &sr, int u, int q, int r1, int K) {
    if (u >= r1) return nullptr;
    if (EPI == EPI_GATEUP || (EPI == EPI_LM && !TIED)) return (q < 4 ? sr.p0 : sr.p1) + (long long)u * K;
    if (EPI == EPI_QKV) {
        if (u < sr.b1) return sr.p0 + (long long)u * K;
        if (u < sr.b2) return sr.p1 + (long long)(u - sr.b1) * K;
        return sr.p2 + (long long)(u - sr.b2) * K;
    }
    return sr.p0 + (long long)u * K;
}

// Units of a CTA's range [r0, r1) are spread over the tile slots: slot q of group g holds
// unit r0 + (q mod GR) * per + g, per = ceil((r1 - r0) / GR), so the 8 copies of a tile
// come from 8 places far apart in memory instead of one contiguous span.
__device__ __forceinline__ int slot_unit(int r0, int per, int GR, int q, int g) { return r0 + (q % GR) * per + g; }

template <typename T, int EPI, bool TIED>
__global__ void __launch_bounds__(TG_THREADS, 1) k_gemv(const Plan *__restrict__ P, int round) {
    extern __shared__ __align__(128) unsigned char tg_smem[];
    constexpr int NRHS = EPI == EPI_LM ? 2 : 1;
    constexpr int VEC = WTraits<T>::VEC;
    // units per tile group: rows, or (gate, up) / (head 0, head 1) row pairs
    constexpr int GR = (EPI == EPI_GATEUP || (EPI == EPI_LM && !TIED)) ? TG_RG / 2 : TG_RG;
    __shared__ __align__(8) uint64_t full[TG_MAXNS], empty[TG_MAXNS];
    __shared__ StageList SL;
    __shared__ float cred[TG_CONSUMERS / 32];
    __shared__ int s_done, s_rows[2], s_last;
    __shared__ float s_bv[2][TG_CONSUMERS / 32];
    __shared__ int s_bi[2][TG_CONSUMERS / 32];
    const DevState *st = P->st;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the first launch of a step follows verification, which rewrites the slot state: it
    // waits before reading it; every later launch of the step reads the (stable) state and
    // starts streaming weights before its predecessor has finished
    const bool wait_first = EPI == EPI_QKV && round == 0;
    if (wait_first) {
        pdl_wait();
        pdl_trigger();
    }
    if (warp == 0) {
        if (EPI == EPI_LM) {
            // exit slot (stage n-1 occupied?) and the draft module's newest row
            const int n = P->n, ns = n + 1, head = st->head;
            const bool v = lane < n && st->valid[ring(head, lane, ns)] != 0;
            const unsigned mask = __ballot_sync(0xffffffffu, v);
            if (lane == 0) {
                s_done = st->done;
                s_rows[0] = (mask >> (n - 1)) & 1u ? ring(head, n - 1, ns) : -1;
                s_rows[1] = (pdm_pending(P, st) ? 1 : 0) + __popc(mask) - 1;
                SL.m = 1;
                SL.stage[0] = SL.slot[0] = SL.layer[0] = 0;
            }
        } else {
            warp_stage_list(P, round, SL, &s_done);
        }
        if (lane == 0) {
            for (int i = 0; i < TG_MAXNS; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], TG_CONSUMERS / 32);
            }
            fence_mbar_init();
        }
    }
    __syncthreads();
    if (s_done || SL.m == 0) return;

    const int d = P->d;
    const int N = EPI == EPI_QKV ? P->qkv_rows : EPI == EPI_GATEUP ? P->F : EPI == EPI_LM ? P->V : d;
    const int K = (EPI == EPI_QKV || EPI == EPI_GATEUP || EPI == EPI_LM) ? d : (EPI == EPI_OPROJ ? P->q_rows : P->F);
    const int nch = (int)(((long long)K * sizeof(T) + TG_ROWB - 1) / TG_ROWB);
    const int KC = ((K + nch - 1) / nch + VEC - 1) / VEC * VEC;
    // shared memory: x (NRHS x K floats) first, then the ring of 8-row tiles
    // (the O projection also keeps the attention merge weights, 2 x Hq x chunks floats, after x)
    const int xfloats = NRHS * K + (EPI == EPI_OPROJ ? 2 * P->Hq * P->att_max_chunks : 0);
    const int xbytes = (xfloats * (int)sizeof(float) + 127) / 128 * 128;
    const int rowb = (KC * (int)sizeof(T) + 127) / 128 * 128;
    const int stage_bytes = TG_RG * rowb;
    const int NS = min(TG_MAXNS, (TG_SMEM - xbytes) / stage_bytes);
    float *xs = reinterpret_cast<float *>(tg_smem);
    unsigned char *stages = tg_smem + xbytes;
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
                const SegRows<T> sr = seg_rows<T, EPI, TIED>(P, P->tl[SL.layer[i]]);
                const int per = (r1 - r0 + GR - 1) / GR;
                for (int g = 0; g < per; ++g) {
                    const T *rp[TG_RG];
                    int nrows = 0;
#pragma unroll
                    for (int q = 0; q < TG_RG; ++q) {
                        rp[q] = tile_row<T, EPI, TIED>(sr, slot_unit(r0, per, GR, q, g), q, r1, K);
                        nrows += rp[q] != nullptr;
                    }
                    for (int c = 0; c < nch; ++c) {
                        const int kc0 = c * KC, len = min(KC, K - kc0);
                        const int sidx = tile % NS;
                        const uint32_t u = tile / NS;
                        if (!mbar_wait(&empty[sidx], (u & 1) ^ 1, P->wait_cycles)) P->st->error = ERR_TIMEOUT;
                        const uint32_t bytes = (uint32_t)len * sizeof(T);
                        // test hook (off unless the handle was created with it): the CTA's very
                        // last tile is never loaded, so its consumers' wait runs out
                        if (EPI == EPI_GATEUP && P->test_withhold && blockIdx.x == 0 && round == 0 && c == nch - 1 &&
                            g == per - 1 && (long long)(i + 1) * N >= hi && P->st->t == 0) {
                            ++tile;
                            continue;
                        }
                        mbar_expect_tx(&full[sidx], bytes * nrows);
#pragma unroll
                        for (int q = 0; q < TG_RG; ++q)
                            if (rp[q]) bulk_g2s(stages + sidx * stage_bytes + q * rowb, rp[q] + kc0, bytes, &full[sidx]);
                        ++tile;
                    }
                }
                r = (long long)(i + 1) * N;
            }
        }
        return;
    }

    // ------------------------------ consumers -----------------------------------------
    if (!wait_first) {
        pdl_wait();   // the inputs staged below come from the preceding launch
        pdl_trigger();
    }
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
        if (EPI == EPI_QKV) c_stage_norm<T>(P->X + (long long)slot * d, w.g1, d, P->eps, xs, cred);
        else if (EPI == EPI_GATEUP) c_stage_norm<T>(P->X + (long long)slot * d, w.g2, d, P->eps, xs, cred);
        else if (EPI == EPI_OPROJ) {
            c_stage_attn<T>(P, s, SL.pos[i], xs, xs + K);
        } else if (EPI == EPI_DOWN) {
            c_stage_swiglu<T>(P->U + (long long)s * 2 * P->F, xs, K);
            named_sync(BAR_C, TG_CONSUMERS);
        } else {
            if (s_rows[0] >= 0) c_stage_norm<T>(P->X + (long long)s_rows[0] * d, P->gf, d, P->eps, xs, cred);
            else {
                for (int k = tid; k < d; k += TG_CONSUMERS) xs[k] = 0.f;
                named_sync(BAR_C, TG_CONSUMERS);
            }
            if (P->Ls > 0) c_stage_norm<T>(P->Xp + (long long)s_rows[1] * d, P->pdm_gf, d, P->eps, xs + d, cred);
            else {
                for (int k = tid; k < d; k += TG_CONSUMERS) xs[d + k] = 0.f;
                named_sync(BAR_C, TG_CONSUMERS);
            }
        }
        const int per = (r1 - r0 + GR - 1) / GR;
        // tied LM head with one piece per row: warp q takes slot q of two consecutive tiles at
        // once and reads each x vector once for both rows (the two right-hand sides make the
        // head otherwise bound by shared-memory reads of x)
        const bool pair = EPI == EPI_LM && TIED && nch == 1 && NS >= 2;
        if constexpr (EPI == EPI_LM && TIED) {
            if (pair) {
                const int q = warp, plane = d >> 1, nvec = K / VEC;
                for (int g = 0; g < per; g += 2) {
                    const bool two = g + 1 < per;
                    const int uA = slot_unit(r0, per, GR, q, g), uB = slot_unit(r0, per, GR, q, g + 1);
                    const bool rvA = uA < r1, rvB = two && uB < r1;
                    const int sA = tile % NS, sB = (tile + 1) % NS;
                    if (!mbar_wait(&full[sA], (tile / NS) & 1, P->wait_cycles)) P->st->error = ERR_TIMEOUT;
                    if (two && !mbar_wait(&full[sB], ((tile + 1) / NS) & 1, P->wait_cycles)) P->st->error = ERR_TIMEOUT;
                    const unsigned char *tA = stages + sA * stage_bytes + q * rowb;
                    const unsigned char *tB = stages + sB * stage_bytes + q * rowb;
                    float cA = 0.f, eA = 0.f, cB = 0.f, eB = 0.f;
                    for (int v = lane; v < nvec; v += 32) {
                        XV<T> xa, xb;
                        xa.load(xs, v * VEC, plane);
                        xb.load(xs + d, v * VEC, plane);
                        if (rvA) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(tA + v * 16);
                            cA = xa.dot(w, cA);
                            eA = xb.dot(w, eA);
                        }
                        if (rvB) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(tB + v * 16);
                            cB = xa.dot(w, cB);
                            eB = xb.dot(w, eB);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[sA]);
                        if (two) mbar_arrive(&empty[sB]);
                    }
                    tile += two ? 2 : 1;
                    cA = warp_sum(cA);
                    eA = warp_sum(eA);
                    cB = warp_sum(cB);
                    eB = warp_sum(eB);
                    if (lane == 0) {
                        for (int k = 0; k < 2; ++k) {
                            const bool rvk = k == 0 ? rvA : rvB;
                            if (!rvk) continue;
                            const int unit = k == 0 ? uA : uB;
                            const float z0 = k == 0 ? cA : cB, z1 = k == 0 ? eA : eB;
                            P->logits[unit] = z0;
                            P->logits[(long long)P->V + unit] = z1;
                            if (dl) dl[unit] = z1;
                            if (z0 > bv[0] || (z0 == bv[0] && unit < bi[0])) {
                                bv[0] = z0;
                                bi[0] = unit;
                            }
                            if (z1 > bv[1] || (z1 == bv[1] && unit < bi[1])) {
                                bv[1] = z1;
                                bi[1] = unit;
                            }
                        }
                    }
                }
                r = (long long)(i + 1) * N;
                continue;
            }
        }
        for (int g = 0; g < per; ++g) {
            // warp q owns tile slot q for all chunks of this group
            const int q = warp;
            const int unit = slot_unit(r0, per, GR, q, g);
            const bool rv = unit < r1;
            // the residual this row adds to, loaded before the dot product so that its latency
            // overlaps the tile instead of stalling the warp after it
            float xold = 0.f, gfin = 0.f;
            if ((EPI == EPI_OPROJ || EPI == EPI_DOWN) && lane == 0 && rv) xold = P->X[(long long)slot * d + unit];
            // the last layer's output is also the LM head's bf16 input row x * g_final
            const bool lm_row = EPI == EPI_DOWN && sizeof(T) == 2 && layer + 1 == P->L;
            if (lm_row && lane == 0 && rv) gfin = P->gf[unit];
            float acc0 = 0.f, acc1 = 0.f;
            for (int c = 0; c < nch; ++c) {
                const int kc0 = c * KC, len = min(KC, K - kc0);
                const int sidx = tile % NS;
                const uint32_t u = tile / NS;
                if (!mbar_wait(&full[sidx], u & 1, P->wait_cycles)) P->st->error = ERR_TIMEOUT;
                if (rv) {
                    const unsigned char *tb = stages + sidx * stage_bytes + q * rowb;
                    const int nvec = len / VEC;
                    // x of this chunk (and of the second right-hand side for the LM head)
                    const int Kx = EPI == EPI_LM ? d : K, plane = Kx >> 1;
                    const float *xa = xs + (EPI == EPI_LM && !TIED && q >= 4 ? d : 0);
                    const float *xb = xs + d;
                    // vectors lane, lane+32, ... alternate between two accumulator chains
                    // (fixed order: results do not depend on anything but the row and x)
                    float c0 = 0.f, c1 = 0.f, e0 = 0.f, e1 = 0.f;
                    int v = lane;
                    for (; v + 32 < nvec; v += 64) {
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(tb + v * 16);
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(tb + (v + 32) * 16);
                        const int f0 = kc0 + v * VEC, f1 = f0 + 32 * VEC;
                        c0 = dot_x<T>(w0, xa, f0, plane, c0);
                        c1 = dot_x<T>(w1, xa, f1, plane, c1);
                        if (EPI == EPI_LM && TIED) {
                            e0 = dot_x<T>(w0, xb, f0, plane, e0);
                            e1 = dot_x<T>(w1, xb, f1, plane, e1);
                        }
                    }
                    if (v < nvec) {
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(tb + v * 16);
                        c0 = dot_x<T>(w0, xa, kc0 + v * VEC, plane, c0);
                        if (EPI == EPI_LM && TIED) e0 = dot_x<T>(w0, xb, kc0 + v * VEC, plane, e0);
                    }
                    acc0 += c0 + c1;
                    if (EPI == EPI_LM && TIED) acc1 += e0 + e1;
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
                    P->X[(long long)slot * d + unit] = xold + acc0;
                } else if (EPI == EPI_GATEUP) {
                    // raw gate (rows 0..3) and up (rows 4..7) sums; SiLU(gate) * up is formed when
                    // the down projection stages its input
                    P->U[(long long)s * 2 * P->F + (q < 4 ? 0 : P->F) + unit] = acc0;
                } else if (EPI == EPI_DOWN) {
                    const float xn = xold + acc0;
                    P->X[(long long)slot * d + unit] = xn;
                    const int a = P->aidx[layer + 1];
                    if (a >= 0) {
                        P->ANCH[((long long)slot * P->nB + a) * d + unit] = xn;
                        if (sizeof(T) == 2) {
                            // the draft projection's input in two bf16 parts (value, remainder)
                            const __nv_bfloat16 hb = __float2bfloat16_rn(xn);
                            const long long ai = ((long long)slot * P->nB + a) * d + unit;
                            P->ANCHb[ai] = hb;
                            P->ANCHb[(long long)(P->n + 1) * P->nB * d + ai] = __float2bfloat16_rn(xn - __bfloat162float(hb));
                        }
                    }
                    if (lm_row) {
                        // the LM head's input row in two bf16 parts: the value and the rest
                        const float xl = xn * gfin;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(xl);
                        P->Xlm[unit] = hi;
                        P->Xlm[2 * d + unit] = __float2bfloat16_rn(xl - __bfloat162float(hi));
                    }
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
static int smem_for(const Plan &, int) { return TG_SMEM; }

template <typename T, int EPI>
static void launch_epi(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    launch_k(k_gemv<T, EPI, true>, dim3(grid), dim3(TG_THREADS), smem_for(h, EPI), s, h.pdl != 0, P, round);
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
    if (lm_on_tensor_cores(h)) {
        launch_pdm_lm<T>(P, h, grid, s);
        return;
    }
    if (h.pdm_lm_head == h.lm_head)
        launch_k(k_gemv<T, EPI_LM, true>, dim3(grid), dim3(TG_THREADS), smem_for(h, EPI_LM), s, h.pdl != 0, P, 0);
    else
        launch_k(k_gemv<T, EPI_LM, false>, dim3(grid), dim3(TG_THREADS), smem_for(h, EPI_LM), s, h.pdl != 0, P, 0);
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
