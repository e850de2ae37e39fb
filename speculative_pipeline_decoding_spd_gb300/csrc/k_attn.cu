// Decode attention of one pipeline step.
//
// Target mode: each occupied stage's token attends, in the layer its stage runs at this
// round, to KV positions 0..pos (machine review "The reading": the n tokens of one
// sequence advance in parallel; the staircase guarantees that every earlier position
// already holds this layer's K,V).  RoPE of q and k and the KV append at pos are fused
// here; the QKV GEMV leaves raw projections.
// Draft mode: the draft module's rows (consecutive positions) attend causally to its
// own KV cache, whose entries for the rows were written by the QKV epilogue.
//
// Split-K over fixed 128-position chunks: one CTA per (problem, kv head, chunk) holds
// the whole GQA group; the last CTA of a (problem, kv head) merges the chunks in chunk
// order.  Chunk boundaries do not depend on the problem mix, so results are identical
// whatever stages share the launch.
#include "common.cuh"

namespace spd {

constexpr int ATT_THREADS = 128;
constexpr int ATT_MAXG = 8;     // query heads per kv head
constexpr int ATT_MAXHD = 128;

template <typename T>
__device__ __forceinline__ void load_dims(const T *p, int lane, int dpl, float *out) {
    for (int e = 0; e < dpl; ++e) out[e] = WTraits<T>::get(p, lane * dpl + e);
}
template <>
__device__ __forceinline__ void load_dims<__nv_bfloat16>(const __nv_bfloat16 *p, int lane, int dpl, float *out) {
    if (dpl == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p + lane * 4);
        out[0] = bf_lo(u.x);
        out[1] = bf_hi(u.x);
        out[2] = bf_lo(u.y);
        out[3] = bf_hi(u.y);
    } else {
        for (int e = 0; e < dpl; ++e) out[e] = __bfloat162float(p[lane * dpl + e]);
    }
}

template <typename T, bool TARGET>
__global__ void __launch_bounds__(ATT_THREADS) k_attn(const Plan *__restrict__ P, int arg) {
    __shared__ __align__(16) float qs[ATT_MAXG][ATT_MAXHD];
    __shared__ float sc[ATT_MAXG][ATT_CHUNK];
    __shared__ float knew[ATT_MAXHD], vnew[ATT_MAXHD];
    __shared__ float opart[ATT_THREADS / 32][ATT_MAXG];
    __shared__ float s_m[ATT_MAXG], s_l[ATT_MAXG];
    __shared__ int s_ok, s_pos, s_layer, s_src, s_out, s_last;
    const int Hkv = P->Hkv, hd = P->hd, G = P->Hq / Hkv, half = hd / 2;
    const int g = blockIdx.x % Hkv, c = blockIdx.x / Hkv, prob = blockIdx.y;
    const DevState *st = P->st;
    if (threadIdx.x == 0) {
        int ok = !st->done;
        int pos = 0, layer = 0, src = 0, out = 0;
        if (ok && TARGET) {
            const int n = P->n, ns = n + 1, head = st->head;
            int m = 0;
            ok = 0;
            for (int s = 0; s < n; ++s) {
                const int slot = ring(head, s, ns);
                if (!st->valid[slot]) continue;
                const int l = P->b[s] + arg;
                if (l >= P->b[s + 1]) continue;
                if (m == prob) {
                    ok = 1;
                    pos = st->pos[slot];
                    layer = l;
                    src = s;
                    out = s;
                }
                ++m;
            }
        } else if (ok) {
            PdmRows pr;
            build_pdm_rows(P, pr);
            ok = prob < pr.R;
            pos = pr.pos0 + prob;
            layer = arg;
            src = prob;
            out = prob;
        }
        if (ok && c * ATT_CHUNK > pos) ok = 0;
        s_ok = ok;
        s_pos = pos;
        s_layer = layer;
        s_src = src;
        s_out = out;
    }
    __syncthreads();
    if (!s_ok) return;
    const int pos = s_pos, S = pos + 1, nch = (S + ATT_CHUNK - 1) / ATT_CHUNK;
    const int j0 = c * ATT_CHUNK, cnt = min(ATT_CHUNK, S - j0);
    const long long kvoff = TARGET ? (long long)s_layer * P->kv_stride : (long long)s_layer * P->kv_stride;
    const T *Kc = reinterpret_cast<const T *>(TARGET ? P->kc : P->pkc) + kvoff;
    const T *Vc = reinterpret_cast<const T *>(TARGET ? P->vc : P->pvc) + kvoff;
    const long long rowstride = (long long)Hkv * hd;
    const bool owner = TARGET && (c == nch - 1);

    // ---- q (and k_new, v_new) for this kv head
    if (TARGET) {
        const float *raw = P->QKV + (long long)s_src * P->qkv_rows;
        const float2 *cs = P->rope + (long long)pos * half;
        for (int idx = threadIdx.x; idx < G * half; idx += blockDim.x) {
            const int h = idx / half, i = idx % half;
            const float *qh = raw + (long long)(g * G + h) * hd;
            const float2 r = cs[i];
            const float a = qh[i], b = qh[i + half];
            qs[h][i] = a * r.x - b * r.y;
            qs[h][i + half] = b * r.x + a * r.y;
        }
        if (owner) {
            const float *kh = raw + P->q_rows + (long long)g * hd;
            const float *vh = raw + P->q_rows + P->kv_rows + (long long)g * hd;
            T *kdst = reinterpret_cast<T *>(P->kc) + kvoff + (long long)pos * rowstride + (long long)g * hd;
            T *vdst = reinterpret_cast<T *>(P->vc) + kvoff + (long long)pos * rowstride + (long long)g * hd;
            for (int i = threadIdx.x; i < half; i += blockDim.x) {
                const float2 r = cs[i];
                const float a = kh[i], b = kh[i + half];
                const auto k0 = WTraits<T>::store(a * r.x - b * r.y);
                const auto k1 = WTraits<T>::store(b * r.x + a * r.y);
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
    } else {
        const float *q = P->QKVp + (long long)s_src * P->qkv_rows;
        for (int idx = threadIdx.x; idx < G * hd; idx += blockDim.x) {
            const int h = idx / hd, i = idx % hd;
            qs[h][i] = q[(long long)(g * G + h) * hd + i];
        }
    }
    __syncthreads();

    // ---- scores for this chunk: one warp per position, lanes split the head dim
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int dpl = hd / 32;
    const float scale = P->scale;
    for (int j = warp; j < cnt; j += ATT_THREADS / 32) {
        const int p = j0 + j;
        float kv[ATT_MAXHD / 32];
        if (owner && p == pos) {
            for (int e = 0; e < dpl; ++e) kv[e] = knew[lane * dpl + e];
        } else {
            load_dims<T>(Kc + (long long)p * rowstride + (long long)g * hd, lane, dpl, kv);
        }
        for (int h = 0; h < G; ++h) {
            float part = 0.f;
            for (int e = 0; e < dpl; ++e) part = fmaf(qs[h][lane * dpl + e], kv[e], part);
            part = warp_sum(part);
            if (lane == 0) sc[h][j] = part * scale;
        }
    }
    __syncthreads();
    // ---- chunk softmax per head
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float m = -INFINITY;
        for (int j = lane; j < cnt; j += 32) m = fmaxf(m, sc[h][j]);
        m = warp_max(m);
        float l = 0.f;
        for (int j = lane; j < cnt; j += 32) {
            const float e = expf(sc[h][j] - m);
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
    // ---- o = sum_j p_j v_j : thread = (dim, parity)
    const int npar = ATT_THREADS / hd;   // 1 (hd=128) or 2 (hd=64)
    const int dim = threadIdx.x % hd, par = threadIdx.x / hd;
    float o[ATT_MAXG];
    for (int h = 0; h < ATT_MAXG; ++h) o[h] = 0.f;
    if (par < npar) {
        for (int j = par; j < cnt; j += npar) {
            const int p = j0 + j;
            const float v = (owner && p == pos) ? vnew[dim] : WTraits<T>::get(Vc, (long long)p * rowstride + (long long)g * hd + dim);
            for (int h = 0; h < G; ++h) o[h] = fmaf(sc[h][j], v, o[h]);
        }
    }
    __shared__ float opar[2][ATT_MAXG][ATT_MAXHD];
    if (npar > 1) {
        if (par < 2)
            for (int h = 0; h < G; ++h) opar[par][h][dim] = o[h];
        __syncthreads();
        if (par == 0)
            for (int h = 0; h < G; ++h) o[h] = opar[0][h][dim] + opar[1][h][dim];
    }
    float *outp = (TARGET ? P->ATT : P->ATTp) + (long long)s_out * P->q_rows;
    if (nch == 1) {
        if (par == 0)
            for (int h = 0; h < G; ++h) outp[(long long)(g * G + h) * hd + dim] = o[h] / s_l[h];
        return;
    }
    float *part = TARGET ? P->att_part : P->patt_part;
    int *cntp = (TARGET ? P->att_cnt : P->patt_cnt) + prob * Hkv + g;
    const int maxch = P->att_max_chunks;
    auto pidx = [&](int h, int cc) -> long long {
        return (((long long)prob * P->Hq + g * G + h) * maxch + cc) * (hd + 2);
    };
    if (par == 0) {
        for (int h = 0; h < G; ++h) {
            part[pidx(h, c) + dim] = o[h];
            if (dim == 0) {
                part[pidx(h, c) + hd] = s_m[h];
                part[pidx(h, c) + hd + 1] = s_l[h];
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(cntp, 1) == nch - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (par == 0) {
        for (int h = 0; h < G; ++h) {
            float M = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(part + pidx(h, cc) + hd));
            float num = 0.f, den = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
                const float w = expf(__ldcg(part + pidx(h, cc) + hd) - M);
                num = fmaf(w, __ldcg(part + pidx(h, cc) + dim), num);
                den = fmaf(w, __ldcg(part + pidx(h, cc) + hd + 1), den);
            }
            outp[(long long)(g * G + h) * hd + dim] = num / den;
        }
    }
    if (threadIdx.x == 0) *cntp = 0;
}

template <typename T>
void launch_target_attn(const Plan *P, const Plan &h, int round, cudaStream_t s) {
    dim3 grid(h.att_max_chunks * h.Hkv, h.n);
    k_attn<T, true><<<grid, ATT_THREADS, 0, s>>>(P, round);
}
template <typename T>
void launch_pdm_attn(const Plan *P, const Plan &h, int layer, cudaStream_t s) {
    dim3 grid(h.att_max_chunks * h.Hkv, h.n + 1);
    k_attn<T, false><<<grid, ATT_THREADS, 0, s>>>(P, layer);
}

template void launch_target_attn<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_target_attn<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_attn<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_attn<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);

}  // namespace spd
