// Decode attention device code shared by the pipeline step (k_attn.cu) and the
// standalone attention entry points (k_ops.cu).
//
// Split-K over fixed 128-position chunks: one CTA of 256 threads per (problem, kv head,
// chunk) holds the whole GQA group.  Latency is what bounds this kernel (a decode step
// reads a few MB of K/V spread over hundreds of CTAs), so every global access is issued
// as early as possible and all of a thread's loads are in flight together:
//   * the chunk's K and V rows go to shared memory by asynchronous 16-byte copies (no
//     registers held while they are in flight), q is staged (and rotated) meanwhile; fp32
//     rows (the pipeline's caches) share one buffer: K first, V once the scores are done;
//   * scores: thread = (position, head parity), 16-byte K reads from a row pitch that
//     puts 8 consecutive rows on distinct banks, q broadcast from shared memory;
//   * softmax per head in one warp, then o = sum_j p_j v_j with thread = (16-byte vector
//     of the row, position group), 4 heads per pass; position groups are added by a fixed
//     shuffle tree inside a warp, the warps in warp order through shared memory;
//   * the chunk's (o, max, sum) go to the partial buffer; the last CTA of a (problem, kv
//     head) merges the chunks in chunk order with all loads in flight (or, without
//     arrival counters, the consumer of the output merges them).
// Chunk boundaries depend only on the position and each reduction has a fixed order, so
// the result does not depend on what else shares a launch.
#pragma once

#include "common.cuh"

namespace spd {

constexpr int ATT_THREADS = 256;
constexpr int ATT_MAXG = 8;     // query heads per kv head
constexpr int ATT_MAXHD = 128;
constexpr int ATT_HB = 4;       // heads per weighted-sum pass
// CTAs per SM the register budget is sized for: one wave for 8 stages x 8 kv heads of a
// 2K-position context
template <typename T> __host__ __device__ constexpr int att_min_blocks() { return sizeof(T) == 2 ? 3 : 2; }
// fp32 rows: K and V of a chunk take turns in one buffer (the V rows are copied in once the
// scores are done), so that two CTAs fit on an SM and one's copies overlap the other's work
template <typename T> __host__ __device__ constexpr bool att_onebuf() { return sizeof(T) == 4; }

// K and V rows live in shared memory as 32-bit words: 16-bit pairs (T = fp16 or bf16) or
// floats.  lo / hi widen the first / second element of a pair.
template <typename T> struct KVW;
template <> struct KVW<__nv_bfloat16> {
    static constexpr int PER = 2;   // elements per word
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        const __nv_bfloat16 x = __float2bfloat16_rn(a), y = __float2bfloat16_rn(b);
        return (uint32_t)__bfloat16_as_ushort(x) | ((uint32_t)__bfloat16_as_ushort(y) << 16);
    }
    __device__ static __forceinline__ float lo(uint32_t u) { return bf_lo(u); }
    __device__ static __forceinline__ float hi(uint32_t u) { return bf_hi(u); }
};
template <> struct KVW<__half> {
    static constexpr int PER = 2;
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        const __half x = __float2half_rn(a), y = __float2half_rn(b);
        return (uint32_t)__half_as_ushort(x) | ((uint32_t)__half_as_ushort(y) << 16);
    }
    __device__ static __forceinline__ float lo(uint32_t u) { return h_lo(u); }
    __device__ static __forceinline__ float hi(uint32_t u) { return h_hi(u); }
};
template <> struct KVW<float> {
    static constexpr int PER = 1;
};

template <typename T>
__host__ __device__ constexpr int att_words(int hd) { return hd / KVW<T>::PER; }
// row pitch in words: 16 bytes more than the row, so the 16-byte reads of 8 consecutive
// rows at one column fall on 8 distinct 16-byte bank groups
template <typename T>
__host__ __device__ constexpr int att_pitch(int hd) { return att_words<T>(hd) + 4; }

// dynamic shared memory (bytes): Ks [CHUNK][pitch] | Vs [CHUNK][pitch] words (one buffer for
// both with fp32 rows), then qs [G][hd] and the scores [G][CHUNK] as floats.  The per-warp
// weighted sums [8 warps][ATT_HB][hd] floats (16 KB at hd 128) lie over the K rows after the
// scores, or after the scores with fp32 rows (the V rows occupy the K rows there).
template <typename T>
__host__ __device__ constexpr int att_smem_bytes(int hd, int G) {
    return (att_onebuf<T>() ? 1 : 2) * ATT_CHUNK * att_pitch<T>(hd) * 4 + G * hd * 4 + G * ATT_CHUNK * 4 +
           (att_onebuf<T>() ? (ATT_THREADS / 32) * ATT_HB * hd * 4 : 0);
}

// One attention problem: a single query token of Hq heads against cache positions
// 0..S-1 of one layer.
template <typename T>
struct AttnArgs {
    const float *q;          // [Hq][hd] fp32 (raw if rope != nullptr)
    const float2 *rope;      // (cos, sin)[hd/2] at position S-1, or nullptr (q already rotated)
    const float *kraw;       // [Hkv][hd] raw k of position S-1 to rotate and append, or nullptr
    const float *vraw;       // [Hkv][hd] v of position S-1 to append (with kraw)
    T *kc;                   // layer cache base [max_seq][Hkv][hd]
    T *vc;
    int S;                   // attended positions 0..S-1
    float *out;              // [Hq][hd]
    float *part;             // split-K partials [prob][Hq][maxch][att_part_pitch(hd)]
    int *cnt;                // [prob][Hkv] arrival counters (zero between launches), or nullptr:
                             // no merge here, every chunk (even a single one) leaves its partial
    int prob, maxch, Hq, Hkv, hd;
    float scale;
    __nv_bfloat16 *outb;     // if set, the output goes here as two bf16 parts instead of to out:
    long long outb_lo;       // hi at outb[i], lo (what hi left out) at outb[outb_lo + i]
};

template <typename T>
__device__ __forceinline__ void attn_store_out(const AttnArgs<T> &a, long long i, float v) {
    if (a.outb) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        a.outb[i] = hi;
        a.outb[a.outb_lo + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
    } else {
        a.out[i] = v;
    }
}

// The work of CTA (kv head g, chunk c) for one problem, plus the merge when this CTA is
// the last of its (problem, kv head).  Block-uniform: every thread of the CTA calls it.
template <typename T>
__device__ void attn_cta(const AttnArgs<T> &a, int g, int c) {
    extern __shared__ __align__(16) uint32_t kv_smem[];
    __shared__ float knew[ATT_MAXHD], vnew[ATT_MAXHD];
    __shared__ float s_m[ATT_MAXG], s_l[ATT_MAXG];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hd = a.hd, Hkv = a.Hkv, G = a.Hq / Hkv, half = hd / 2;
    const int S = a.S, pos = S - 1, nch = (S + ATT_CHUNK - 1) / ATT_CHUNK;
    const int j0 = c * ATT_CHUNK, cnt = min(ATT_CHUNK, S - j0);
    const long long rowstride = (long long)Hkv * hd;
    const bool owner = a.kraw != nullptr && (c == nch - 1);
    const int W = att_words<T>(hd), KP = att_pitch<T>(hd);
    constexpr bool ONEBUF = att_onebuf<T>();
    uint32_t *Ks = kv_smem, *Vs = ONEBUF ? kv_smem : kv_smem + ATT_CHUNK * KP;
    float *qs = reinterpret_cast<float *>(kv_smem + (ONEBUF ? 1 : 2) * ATT_CHUNK * KP);   // [G][hd]
    float *sc = qs + G * hd;                                       // [G][CHUNK]
    // ---- this chunk's K (and, two buffers, V) rows of kv head g: asynchronous 16-byte copies
    const int vpr = hd * (int)sizeof(T) / 16;   // 16-byte vectors per row
    const long long cbase = ((long long)j0 * rowstride + (long long)g * hd) * (long long)sizeof(T);
    auto copy_rows = [&](uint32_t *dst, const T *src) {
        const char *sb = reinterpret_cast<const char *>(src) + cbase;
        for (int idx = tid; idx < cnt * vpr; idx += ATT_THREADS) {
            const int j = idx / vpr, q = idx - j * vpr;
            cp_async16(dst + j * KP + 4 * q, sb + (long long)j * rowstride * (long long)sizeof(T) + 16 * q);
        }
    };
    copy_rows(Ks, a.kc);
    if (!ONEBUF) copy_rows(Vs, a.vc);
    // ---- the chunk's older positions come from earlier steps; q, k_new and v_new from the
    // preceding launch of this stream
    pdl_wait();
    pdl_trigger();
    // ---- q (rotated here when raw), k_new / v_new appended by the chunk owner
    if (a.rope) {
        for (int idx = tid; idx < G * half; idx += ATT_THREADS) {
            const int h = idx / half, i = idx - h * half;
            const float *qh = a.q + (long long)(g * G + h) * hd;
            const float2 r = a.rope[i];
            const float x0 = qh[i], x1 = qh[i + half];
            qs[h * hd + i] = x0 * r.x - x1 * r.y;
            qs[h * hd + i + half] = x1 * r.x + x0 * r.y;
        }
    } else {
        for (int idx = tid; idx < G * hd; idx += ATT_THREADS) qs[idx] = a.q[(long long)g * G * hd + idx];
    }
    if (owner) {
        const float *kh = a.kraw + (long long)g * hd;
        const float *vh = a.vraw + (long long)g * hd;
        T *kdst = a.kc + (long long)pos * rowstride + (long long)g * hd;
        T *vdst = a.vc + (long long)pos * rowstride + (long long)g * hd;
        if (tid < half) {
            const int i = tid;
            const float2 r = a.rope[i];
            const float x0 = kh[i], x1 = kh[i + half];
            const auto k0 = WTraits<T>::store(x0 * r.x - x1 * r.y);
            const auto k1 = WTraits<T>::store(x1 * r.x + x0 * r.y);
            kdst[i] = k0;
            kdst[i + half] = k1;
            knew[i] = WTraits<T>::get(&k0, 0);
            knew[i + half] = WTraits<T>::get(&k1, 0);
        } else if (tid < half + hd) {
            const int i = tid - half;
            const auto v0 = WTraits<T>::store(vh[i]);
            vdst[i] = v0;
            vnew[i] = WTraits<T>::get(&v0, 0);
        }
    }
    cp_async_wait_all();
    __syncthreads();
    if (owner) {
        // the new position's row comes from this kernel's own (rounded) values
        const int j = pos - j0;
        for (int w = tid; w < W; w += ATT_THREADS) {
            if constexpr (KVW<T>::PER == 2) {
                Ks[j * KP + w] = KVW<T>::pack(knew[2 * w], knew[2 * w + 1]);
                Vs[j * KP + w] = KVW<T>::pack(vnew[2 * w], vnew[2 * w + 1]);
            } else {
                Ks[j * KP + w] = __float_as_uint(knew[w]);
                if (!ONEBUF) Vs[j * KP + w] = __float_as_uint(vnew[w]);
            }
        }
        __syncthreads();
    }

    // ---- scores: thread = (position j, head parity hh); heads hh, hh + 2, ...
    {
        const int j = tid & (ATT_CHUNK - 1), hh = tid / ATT_CHUNK;
        float acc[ATT_MAXG / 2];
#pragma unroll
        for (int u = 0; u < ATT_MAXG / 2; ++u) acc[u] = 0.f;
        if (j < cnt && hh < G) {
            const uint32_t *kr = Ks + j * KP;
            for (int w = 0; w < W; w += 4) {
                const uint4 kw = *reinterpret_cast<const uint4 *>(kr + w);
                float k[8];
                int e0;   // element index of kw.x
                if constexpr (KVW<T>::PER == 2) {
                    k[0] = KVW<T>::lo(kw.x); k[1] = KVW<T>::hi(kw.x); k[2] = KVW<T>::lo(kw.y); k[3] = KVW<T>::hi(kw.y);
                    k[4] = KVW<T>::lo(kw.z); k[5] = KVW<T>::hi(kw.z); k[6] = KVW<T>::lo(kw.w); k[7] = KVW<T>::hi(kw.w);
                    e0 = 2 * w;
                } else {
                    k[0] = __uint_as_float(kw.x); k[1] = __uint_as_float(kw.y);
                    k[2] = __uint_as_float(kw.z); k[3] = __uint_as_float(kw.w);
                    e0 = w;
                }
#pragma unroll
                for (int u = 0; u < ATT_MAXG / 2; ++u) {
                    const int h = hh + 2 * u;
                    if (h < G) {
                        const float4 q0 = *reinterpret_cast<const float4 *>(qs + h * hd + e0);
                        float s = acc[u];
                        s = fmaf(q0.x, k[0], s); s = fmaf(q0.y, k[1], s); s = fmaf(q0.z, k[2], s); s = fmaf(q0.w, k[3], s);
                        if constexpr (KVW<T>::PER == 2) {
                            const float4 q1 = *reinterpret_cast<const float4 *>(qs + h * hd + e0 + 4);
                            s = fmaf(q1.x, k[4], s); s = fmaf(q1.y, k[5], s); s = fmaf(q1.z, k[6], s); s = fmaf(q1.w, k[7], s);
                        }
                        acc[u] = s;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < ATT_MAXG / 2; ++u) {
            const int h = hh + 2 * u;
            if (h < G) sc[h * ATT_CHUNK + j] = j < cnt ? acc[u] * a.scale : -INFINITY;
        }
    }
    __syncthreads();
    if (ONEBUF) copy_rows(Vs, a.vc);   // every K row has been read: the V rows take their place
    // ---- chunk softmax per head
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float *sh = sc + h * ATT_CHUNK;
        float m = -INFINITY;
        for (int j = lane; j < cnt; j += 32) m = fmaxf(m, sh[j]);
        m = warp_max(m);
        float l = 0.f;
        for (int j = lane; j < ATT_CHUNK; j += 32) {
            const float e = j < cnt ? expf(sh[j] - m) : 0.f;
            sh[j] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            s_m[h] = m;
            s_l[h] = l;
        }
    }
    if (ONEBUF) {
        cp_async_wait_all();
        __syncthreads();
        if (owner)
            for (int w = tid; w < W; w += ATT_THREADS) Vs[(pos - j0) * KP + w] = __float_as_uint(vnew[w]);
    }
    __syncthreads();
    // ---- o = sum_j p_j v_j: thread = (16-byte vector vo of the row, position group qg),
    // positions qg, qg + NQ, ...; ATT_HB heads per pass
    auto pidx = [&](int h, int cc) -> long long {
        return (((long long)a.prob * a.Hq + g * G + h) * a.maxch + cc) * att_part_pitch(hd);
    };
    constexpr int EPV = 16 / (int)sizeof(T);        // elements per vector
    const int LPR = hd / EPV, NQ = ATT_THREADS / LPR;
    const int vo = tid % LPR, qg = tid / LPR;
    float *ored = ONEBUF ? sc + G * ATT_CHUNK : reinterpret_cast<float *>(kv_smem);   // [8 warps][ATT_HB][hd]
    for (int hb = 0; hb < G; hb += ATT_HB) {
        float o[ATT_HB][EPV];
#pragma unroll
        for (int u = 0; u < ATT_HB; ++u)
#pragma unroll
            for (int e = 0; e < EPV; ++e) o[u][e] = 0.f;
        for (int j = qg; j < cnt; j += NQ) {
            const uint4 vw = *reinterpret_cast<const uint4 *>(Vs + j * KP + 4 * vo);
            float v[EPV];
            if constexpr (sizeof(T) == 2) {
                v[0] = KVW<T>::lo(vw.x); v[1] = KVW<T>::hi(vw.x); v[2] = KVW<T>::lo(vw.y); v[3] = KVW<T>::hi(vw.y);
                v[4] = KVW<T>::lo(vw.z); v[5] = KVW<T>::hi(vw.z); v[6] = KVW<T>::lo(vw.w); v[7] = KVW<T>::hi(vw.w);
            } else {
                v[0] = __uint_as_float(vw.x); v[1] = __uint_as_float(vw.y);
                v[2] = __uint_as_float(vw.z); v[3] = __uint_as_float(vw.w);
            }
#pragma unroll
            for (int u = 0; u < ATT_HB; ++u)
                if (hb + u < G) {
                    const float p = sc[(hb + u) * ATT_CHUNK + j];
#pragma unroll
                    for (int e = 0; e < EPV; ++e) o[u][e] = fmaf(p, v[e], o[u][e]);
                }
        }
        for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
            for (int u = 0; u < ATT_HB; ++u)
#pragma unroll
                for (int e = 0; e < EPV; ++e) o[u][e] += __shfl_xor_sync(0xffffffffu, o[u][e], off);
        if (hb > 0) __syncthreads();   // the previous pass's sums have been read
        if (lane < LPR) {
#pragma unroll
            for (int u = 0; u < ATT_HB; ++u)
#pragma unroll
                for (int e = 0; e < EPV; ++e) ored[(warp * ATT_HB + u) * hd + vo * EPV + e] = o[u][e];
        }
        __syncthreads();
        for (int idx = tid; idx < ATT_HB * hd; idx += ATT_THREADS) {
            const int u = idx / hd, dd = idx - u * hd, h = hb + u;
            if (h >= G) continue;
            float oo = ored[u * hd + dd];
            for (int w = 1; w < ATT_THREADS / 32; ++w) oo += ored[(w * ATT_HB + u) * hd + dd];
            if (nch == 1 && a.cnt) {
                attn_store_out(a, (long long)(g * G + h) * hd + dd, oo / s_l[h]);
            } else {
                a.part[pidx(h, c) + dd] = oo;
                if (dd == 0) {
                    a.part[pidx(h, c) + hd] = s_m[h];
                    a.part[pidx(h, c) + hd + 1] = s_l[h];
                }
            }
        }
    }
    if (nch == 1 || !a.cnt) return;
    int *cntp = a.cnt + a.prob * Hkv + g;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(cntp, 1) == nch - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // ---- merge in chunk order.  Chunk weights e^{m_c - M}: one warp per head, one lane per
    // chunk (32 at a time, loads in flight together), denominators by a fixed shuffle tree
    // per 32-chunk block added in block order
    float *mw = sc;   // [G][ATT_CHUNK] chunk weights (nch <= ATT_CHUNK)
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float mv[ATT_CHUNK / 32], lv[ATT_CHUNK / 32];
        float M = -INFINITY;
#pragma unroll
        for (int b = 0; b < ATT_CHUNK / 32; ++b) {
            const int cc = b * 32 + lane;
            mv[b] = cc < nch ? __ldcg(a.part + pidx(h, cc) + hd) : -INFINITY;
            lv[b] = cc < nch ? __ldcg(a.part + pidx(h, cc) + hd + 1) : 0.f;
        }
#pragma unroll
        for (int b = 0; b < ATT_CHUNK / 32; ++b) M = fmaxf(M, mv[b]);
        M = warp_max(M);
        float den = 0.f;
#pragma unroll
        for (int b = 0; b < ATT_CHUNK / 32; ++b) {
            const int cc = b * 32 + lane;
            const float w = cc < nch ? expf(mv[b] - M) : 0.f;
            if (cc < nch) mw[h * ATT_CHUNK + cc] = w;
            den += warp_sum(w * lv[b]);
        }
        if (lane == 0) s_l[h] = den;
    }
    __syncthreads();
    for (int idx = tid; idx < G * hd; idx += ATT_THREADS) {
        const int h = idx / hd, dd = idx - h * hd;
        float vals[8];
        float num = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) vals[u] = (c0 + u < nch) ? __ldcg(a.part + pidx(h, c0 + u) + dd) : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + u < nch) num = fmaf(mw[h * ATT_CHUNK + c0 + u], vals[u], num);
        }
        attn_store_out(a, (long long)(g * G + h) * hd + dd, num / s_l[h]);
    }
    if (tid == 0) *cntp = 0;
}

}  // namespace spd
