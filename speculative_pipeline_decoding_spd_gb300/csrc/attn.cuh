// Decode attention device code shared by the pipeline step (k_attn.cu) and the
// standalone attention entry points (k_ops.cu).
//
// Split-K over fixed 128-position chunks: one CTA per (problem, kv head, chunk) holds
// the whole GQA group.  The chunk's K and V rows are staged in shared memory with all
// 16-byte loads in flight, scores are computed one position per thread, the weighted
// sum one (dim pair, position group) per thread.  The last CTA of a (problem, kv head)
// merges the chunks in chunk order.  Chunk boundaries depend only on the position, so
// results do not depend on what else shares a launch.
#pragma once

#include "common.cuh"

namespace spd {

constexpr int ATT_THREADS = 128;
constexpr int ATT_MAXG = 8;     // query heads per kv head
constexpr int ATT_MAXHD = 128;

// K/V tiles live in shared memory as 32-bit words: bf16 pairs (T = bf16) or floats.
template <typename T> struct KVW {
    static constexpr int PER = 2;   // elements per word
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        const __nv_bfloat16 x = __float2bfloat16_rn(a), y = __float2bfloat16_rn(b);
        return (uint32_t)__bfloat16_as_ushort(x) | ((uint32_t)__bfloat16_as_ushort(y) << 16);
    }
};
template <> struct KVW<float> {
    static constexpr int PER = 1;
};

template <typename T>
__host__ __device__ constexpr int att_words(int hd) { return hd / KVW<T>::PER; }

// dynamic shared memory: Ks [CHUNK][words+1] (odd pitch: one-row-per-thread reads hit
// distinct banks), Vs [CHUNK][words]
template <typename T>
__host__ __device__ constexpr int att_smem_bytes(int hd) {
    return (ATT_CHUNK * (att_words<T>(hd) + 1) + ATT_CHUNK * att_words<T>(hd)) * 4;
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
    float *part;             // split-K partials [prob][Hq][maxch][hd+2]
    int *cnt;                // [prob][Hkv] arrival counters (zero between launches)
    int prob, maxch, Hq, Hkv, hd;
    float scale;
};

// The work of CTA (kv head g, chunk c) for one problem, plus the merge when this CTA is
// the last of its (problem, kv head).  Block-uniform: every thread of the CTA calls it.
template <typename T>
__device__ void attn_cta(const AttnArgs<T> &a, int g, int c) {
    extern __shared__ __align__(16) uint32_t kv_smem[];
    __shared__ __align__(16) float qs[ATT_MAXG][ATT_MAXHD];
    __shared__ float sc[ATT_MAXG][ATT_CHUNK];
    __shared__ float knew[ATT_MAXHD], vnew[ATT_MAXHD];
    __shared__ float s_m[ATT_MAXG], s_l[ATT_MAXG];
    __shared__ float ored[4][ATT_MAXG][ATT_MAXHD];
    __shared__ int s_last;
    const int hd = a.hd, Hkv = a.Hkv, G = a.Hq / Hkv, half = hd / 2;
    const int S = a.S, pos = S - 1, nch = (S + ATT_CHUNK - 1) / ATT_CHUNK;
    const int j0 = c * ATT_CHUNK, cnt = min(ATT_CHUNK, S - j0);
    const long long rowstride = (long long)Hkv * hd;
    const bool owner = a.kraw != nullptr && (c == nch - 1);
    const int W = att_words<T>(hd), KP = W + 1;
    uint32_t *Ks = kv_smem, *Vs = kv_smem + ATT_CHUNK * KP;

    // ---- stage this chunk's K and V rows of kv head g (2 x 8 16-byte loads in flight)
    {
        const int vec_per_row = hd * (int)sizeof(T) / 16;
        const int total = cnt * vec_per_row;
        constexpr int U = 8;
        for (int b = threadIdx.x; b < total; b += U * blockDim.x) {
            uint4 kv[U], vv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int idx = b + u * blockDim.x;
                if (idx < total) {
                    const int j = idx / vec_per_row, q = idx - j * vec_per_row;
                    const long long off = (long long)(j0 + j) * rowstride + (long long)g * hd;
                    kv[u] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(a.kc + off) + 16 * q);
                    vv[u] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(a.vc + off) + 16 * q);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int idx = b + u * blockDim.x;
                if (idx < total) {
                    const int j = idx / vec_per_row, q = idx - j * vec_per_row;
                    uint32_t *kd = Ks + j * KP + 4 * q;
                    kd[0] = kv[u].x;
                    kd[1] = kv[u].y;
                    kd[2] = kv[u].z;
                    kd[3] = kv[u].w;
                    *reinterpret_cast<uint4 *>(Vs + j * W + 4 * q) = vv[u];
                }
            }
        }
    }
    // ---- q (rotated here when raw), k_new / v_new appended by the chunk owner
    if (a.rope) {
        for (int idx = threadIdx.x; idx < G * half; idx += blockDim.x) {
            const int h = idx / half, i = idx % half;
            const float *qh = a.q + (long long)(g * G + h) * hd;
            const float2 r = a.rope[i];
            const float x0 = qh[i], x1 = qh[i + half];
            qs[h][i] = x0 * r.x - x1 * r.y;
            qs[h][i + half] = x1 * r.x + x0 * r.y;
        }
    } else {
        for (int idx = threadIdx.x; idx < G * hd; idx += blockDim.x) {
            const int h = idx / hd, i = idx % hd;
            qs[h][i] = a.q[(long long)(g * G + h) * hd + i];
        }
    }
    if (owner) {
        const float *kh = a.kraw + (long long)g * hd;
        const float *vh = a.vraw + (long long)g * hd;
        T *kdst = a.kc + (long long)pos * rowstride + (long long)g * hd;
        T *vdst = a.vc + (long long)pos * rowstride + (long long)g * hd;
        for (int i = threadIdx.x; i < half; i += blockDim.x) {
            const float2 r = a.rope[i];
            const float x0 = kh[i], x1 = kh[i + half];
            const auto k0 = WTraits<T>::store(x0 * r.x - x1 * r.y);
            const auto k1 = WTraits<T>::store(x1 * r.x + x0 * r.y);
            kdst[i] = k0;
            kdst[i + half] = k1;
            knew[i] = (float)k0;
            knew[i + half] = (float)k1;
        }
        for (int i = threadIdx.x; i < hd; i += blockDim.x) {
            const auto v0 = WTraits<T>::store(vh[i]);
            vdst[i] = v0;
            vnew[i] = (float)v0;
        }
    }
    __syncthreads();
    if (owner) {
        // the new position's row comes from this kernel's own (rounded) values
        const int j = pos - j0;
        for (int w = threadIdx.x; w < W; w += blockDim.x) {
            if constexpr (KVW<T>::PER == 2) {
                Ks[j * KP + w] = KVW<T>::pack(knew[2 * w], knew[2 * w + 1]);
                Vs[j * W + w] = KVW<T>::pack(vnew[2 * w], vnew[2 * w + 1]);
            } else {
                Ks[j * KP + w] = __float_as_uint(knew[w]);
                Vs[j * W + w] = __float_as_uint(vnew[w]);
            }
        }
        __syncthreads();
    }

    // ---- scores: thread = position, all heads of the group
    {
        const int j = threadIdx.x;
        float acc[ATT_MAXG];
#pragma unroll
        for (int h = 0; h < ATT_MAXG; ++h) acc[h] = 0.f;
        if (j < cnt) {
            const uint32_t *kr = Ks + j * KP;
            for (int w = 0; w < W; ++w) {
                const uint32_t u = kr[w];
                if constexpr (KVW<T>::PER == 2) {
                    const float k0 = bf_lo(u), k1 = bf_hi(u);
#pragma unroll
                    for (int h = 0; h < ATT_MAXG; ++h)
                        if (h < G) acc[h] = fmaf(qs[h][2 * w + 1], k1, fmaf(qs[h][2 * w], k0, acc[h]));
                } else {
                    const float k0 = __uint_as_float(u);
#pragma unroll
                    for (int h = 0; h < ATT_MAXG; ++h)
                        if (h < G) acc[h] = fmaf(qs[h][w], k0, acc[h]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < ATT_MAXG; ++h)
            if (h < G) sc[h][j] = j < cnt ? acc[h] * a.scale : -INFINITY;
    }
    __syncthreads();
    // ---- chunk softmax per head
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float m = -INFINITY;
        for (int j = lane; j < cnt; j += 32) m = fmaxf(m, sc[h][j]);
        m = warp_max(m);
        float l = 0.f;
        for (int j = lane; j < ATT_CHUNK; j += 32) {
            const float e = j < cnt ? expf(sc[h][j] - m) : 0.f;
            sc[h][j] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            s_m[h] = m;
            s_l[h] = l;
        }
    }
    __syncthreads();
    // ---- o = sum_j p_j v_j : thread = (dim pair, position group); shared-memory reads only
    const int npair = hd / 2;
    const int nq = ATT_THREADS / npair;       // 2 (hd 128) or 4 (hd 64) position groups
    const int dp = threadIdx.x % npair, qg = threadIdx.x / npair;
    float o0[ATT_MAXG], o1[ATT_MAXG];
#pragma unroll
    for (int h = 0; h < ATT_MAXG; ++h) o0[h] = o1[h] = 0.f;
    for (int j = qg; j < cnt; j += nq) {
        float v0, v1;
        if constexpr (KVW<T>::PER == 2) {
            const uint32_t u = Vs[j * W + dp];
            v0 = bf_lo(u);
            v1 = bf_hi(u);
        } else {
            v0 = __uint_as_float(Vs[j * W + 2 * dp]);
            v1 = __uint_as_float(Vs[j * W + 2 * dp + 1]);
        }
#pragma unroll
        for (int h = 0; h < ATT_MAXG; ++h)
            if (h < G) {
                const float p = sc[h][j];
                o0[h] = fmaf(p, v0, o0[h]);
                o1[h] = fmaf(p, v1, o1[h]);
            }
    }
#pragma unroll
    for (int h = 0; h < ATT_MAXG; ++h)
        if (h < G) {
            ored[qg][h][2 * dp] = o0[h];
            ored[qg][h][2 * dp + 1] = o1[h];
        }
    __syncthreads();
    auto pidx = [&](int h, int cc) -> long long {
        return (((long long)a.prob * a.Hq + g * G + h) * a.maxch + cc) * (hd + 2);
    };
    for (int idx = threadIdx.x; idx < G * hd; idx += blockDim.x) {
        const int h = idx / hd, dd = idx % hd;
        float o = ored[0][h][dd];
        for (int q = 1; q < nq; ++q) o += ored[q][h][dd];
        if (nch == 1) {
            a.out[(long long)(g * G + h) * hd + dd] = o / s_l[h];
        } else {
            a.part[pidx(h, c) + dd] = o;
            if (dd == 0) {
                a.part[pidx(h, c) + hd] = s_m[h];
                a.part[pidx(h, c) + hd + 1] = s_l[h];
            }
        }
    }
    if (nch == 1) return;
    int *cntp = a.cnt + a.prob * Hkv + g;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(cntp, 1) == nch - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // ---- merge in chunk order: weights e^{m_c - M} per (head, chunk) staged first, then each
    // thread combines its (head, dim) outputs with 8 chunk loads in flight before the adds
    float *mw = &sc[0][0];   // reuse: [G][ATT_CHUNK] chunk weights (nch <= ATT_CHUNK)
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float M = -INFINITY;
        for (int cc = lane; cc < nch; cc += 32) M = fmaxf(M, __ldcg(a.part + pidx(h, cc) + hd));
        M = warp_max(M);
        float den = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
            const float w = expf(__ldcg(a.part + pidx(h, cc) + hd) - M);
            if (lane == 0) mw[h * ATT_CHUNK + cc] = w;
            den = fmaf(w, __ldcg(a.part + pidx(h, cc) + hd + 1), den);
        }
        if (lane == 0) s_l[h] = den;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * hd; idx += blockDim.x) {
        const int h = idx / hd, dd = idx % hd;
        float vals[8];
        float num = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) vals[u] = (c0 + u < nch) ? __ldcg(a.part + pidx(h, c0 + u) + dd) : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + u < nch) num = fmaf(mw[h * ATT_CHUNK + c0 + u], vals[u], num);
        }
        a.out[(long long)(g * G + h) * hd + dd] = num / s_l[h];
    }
    if (threadIdx.x == 0) *cntp = 0;
}

}  // namespace spd
