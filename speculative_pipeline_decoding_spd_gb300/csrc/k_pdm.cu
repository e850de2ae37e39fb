// Pipeline Draft Module kernels (run on the second stream, concurrently with the
// target's rounds).
//
// Speculative pipeline decoding, machine review "What carries the argument" / "Core
// claim": the module reads the pipeline's INPUT states, concatenates the target's
// hidden states at the anchor depths (deeper anchors of in-flight tokens are not yet
// computed and enter as zeros), projects them to one feature and runs Ls decoder layers
// and the LM head to propose the next token.  Its rows in one step are the token that
// left the pipeline last step (all anchors; its K,V stay in the module's cache) and
// the in-flight tokens, at consecutive positions, so its attention is plain causal
// attention over its own cache.
//
// Every GEMM here multiplies one weight matrix by R <= n+1 row vectors (a skinny
// GEMM), so it runs on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate):
// the weights are the M side streamed straight from HBM with 16-byte loads, the R
// activation rows (bf16 in shared memory) the N side.  The K dimension of one
// product is kept in a permuted order that is the same for both operands, so each
// lane's 16-byte weight load feeds the A fragment directly.  K is split over CTAs; the
// last CTA of a 128-row block adds the partial sums in split order (deterministic) and
// runs the epilogue (RoPE + KV append, residual add, ...); the last block overall
// recomputes the rows' RMS statistics for the next normalisation.
#include "common.cuh"

namespace spd {

enum { XM_FEAT = 0, XM_NORM1, XM_NORM2, XM_ATT, XM_SILU };
enum { SE_PROJ = 0, SE_QKV, SE_OPROJ, SE_GATEUP, SE_DOWN };
constexpr int SK_THREADS = 256;

template <typename T> struct SkX { using type = float; };
template <> struct SkX<__nv_bfloat16> { using type = __nv_bfloat16; };

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename T, int SE>
__device__ __forceinline__ const T *sk_row(const Plan *__restrict__ P, int layer, int row, int K) {
    if (SE == SE_PROJ) return reinterpret_cast<const T *>(P->proj) + (long long)row * K;
    const LayerW &w = P->pl[layer];
    if (SE == SE_QKV) {
        if (row < P->q_rows) return reinterpret_cast<const T *>(w.wq) + (long long)row * K;
        row -= P->q_rows;
        if (row < P->kv_rows) return reinterpret_cast<const T *>(w.wk) + (long long)row * K;
        return reinterpret_cast<const T *>(w.wv) + (long long)(row - P->kv_rows) * K;
    }
    if (SE == SE_OPROJ) return reinterpret_cast<const T *>(w.wo) + (long long)row * K;
    if (SE == SE_GATEUP) {
        if (row < P->F) return reinterpret_cast<const T *>(w.wg) + (long long)row * K;
        return reinterpret_cast<const T *>(w.wu) + (long long)(row - P->F) * K;
    }
    return reinterpret_cast<const T *>(w.wd) + (long long)row * K;
}

template <int XM>
__device__ __forceinline__ float sk_xval(const Plan *__restrict__ P, const PdmRows &pr, int layer, int r, int k) {
    const int d = P->d;
    if (XM == XM_FEAT) {
        const int a = k / d, off = k - a * d;
        if (P->anchors[a] > pr.depth[r]) return 0.f;
        return P->ANCH[((long long)pr.slot[r] * P->nB + a) * d + off];
    }
    if (XM == XM_NORM1 || XM == XM_NORM2) {
        const float *g = XM == XM_NORM1 ? P->pl[layer].g1 : P->pl[layer].g2;
        return (P->Xp[(long long)r * d + k] * P->inv_rms_p[r]) * g[k];
    }
    if (XM == XM_ATT) return P->ATTp[(long long)r * P->q_rows + k];
    const float gg = P->GUp[(long long)r * 2 * P->F + k];
    const float uu = P->GUp[(long long)r * 2 * P->F + P->F + k];
    return silu_f(gg) * uu;
}

template <typename T, int NT, int XM, int SE>
__global__ void __launch_bounds__(SK_THREADS) k_skinny(const Plan *__restrict__ P, int layer, int N, int K, int nks) {
    using XT = typename SkX<T>::type;
    constexpr int RP = NT * 8;
    extern __shared__ __align__(16) unsigned char sk_smem[];
    __shared__ PdmRows pr;
    __shared__ int s_done, s_last, s_glast;
    if (threadIdx.x < 32) warp_pdm_rows(P, pr, &s_done);
    __syncthreads();
    if (s_done) return;
    const int R = pr.R;
    const int nrb = (N + SK_ROWS - 1) / SK_ROWS;
    const int rb = blockIdx.x / nks, ks = blockIdx.x % nks;
    const int nch = K / SK_KCHUNK;
    const int c0 = (int)((long long)nch * ks / nks), c1 = (int)((long long)nch * (ks + 1) / nks);
    const int k0 = c0 * SK_KCHUNK, kseg = (c1 - c0) * SK_KCHUNK;
    const int kmax = ((nch + nks - 1) / nks) * SK_KCHUNK;
    const int pitch = kmax + (sizeof(XT) == 2 ? 32 : 4);   // elements; keeps 16-byte rows off one bank
    XT *xs = reinterpret_cast<XT *>(sk_smem);

    // ---- stage the R activation rows of this K segment (8 loads in flight per thread)
    const int total = RP * kseg;
    for (int b = threadIdx.x; b < total; b += 8 * blockDim.x) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = b + u * blockDim.x;
            const int r = idx / kseg, kk = idx - r * kseg;
            v[u] = (idx < total && r < R) ? sk_xval<XM>(P, pr, layer, r, k0 + kk) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = b + u * blockDim.x;
            if (idx >= total) continue;
            const int r = idx / kseg, kk = idx - r * kseg;
            if (sizeof(XT) == 2)
                reinterpret_cast<__nv_bfloat16 *>(xs)[r * pitch + kk] = __float2bfloat16_rn(v[u]);
            else
                reinterpret_cast<float *>(xs)[r * pitch + kk] = v[u];
        }
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rbase = rb * SK_ROWS + warp * 16;
    float *part = P->sk_part;
    if constexpr (sizeof(XT) == 2) {
        // tensor-core engine
        const int gq = lane >> 2, tq = lane & 3;
        const int ra = min(rbase + gq, N - 1), rc = min(rbase + gq + 8, N - 1);
        const T *wa = sk_row<T, SE>(P, layer, ra, K) + k0 + 8 * tq;
        const T *wc = sk_row<T, SE>(P, layer, rc, K) + k0 + 8 * tq;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(xs) + 8 * tq;
        const bool active = rbase < N;
        int kk = 0;
        if (active) {
            for (; kk + 2 * SK_KCHUNK <= kseg; kk += 2 * SK_KCHUNK) {
                uint4 A[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    A[h][0] = ld_stream(wa + kk + h * SK_KCHUNK);
                    A[h][1] = ld_stream(wc + kk + h * SK_KCHUNK);
                    A[h][2] = ld_stream(wa + kk + h * SK_KCHUNK + 32);
                    A[h][3] = ld_stream(wc + kk + h * SK_KCHUNK + 32);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const __nv_bfloat16 *xr = xb + (nt * 8 + gq) * pitch + kk + h * SK_KCHUNK;
                        const uint4 b0 = *reinterpret_cast<const uint4 *>(xr);
                        const uint4 b1 = *reinterpret_cast<const uint4 *>(xr + 32);
                        mma_bf16(acc[nt], A[h][0].x, A[h][1].x, A[h][0].y, A[h][1].y, b0.x, b0.y);
                        mma_bf16(acc[nt], A[h][0].z, A[h][1].z, A[h][0].w, A[h][1].w, b0.z, b0.w);
                        mma_bf16(acc[nt], A[h][2].x, A[h][3].x, A[h][2].y, A[h][3].y, b1.x, b1.y);
                        mma_bf16(acc[nt], A[h][2].z, A[h][3].z, A[h][2].w, A[h][3].w, b1.z, b1.w);
                    }
                }
            }
            for (; kk < kseg; kk += SK_KCHUNK) {
                const uint4 a0 = ld_stream(wa + kk), a1 = ld_stream(wc + kk);
                const uint4 a2 = ld_stream(wa + kk + 32), a3 = ld_stream(wc + kk + 32);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const __nv_bfloat16 *xr = xb + (nt * 8 + gq) * pitch + kk;
                    const uint4 b0 = *reinterpret_cast<const uint4 *>(xr);
                    const uint4 b1 = *reinterpret_cast<const uint4 *>(xr + 32);
                    mma_bf16(acc[nt], a0.x, a1.x, a0.y, a1.y, b0.x, b0.y);
                    mma_bf16(acc[nt], a0.z, a1.z, a0.w, a1.w, b0.z, b0.w);
                    mma_bf16(acc[nt], a2.x, a3.x, a2.y, a3.y, b1.x, b1.y);
                    mma_bf16(acc[nt], a2.z, a3.z, a2.w, a3.w, b1.z, b1.w);
                }
            }
            // D fragment: (row gq, cols 2tq, 2tq+1) and (row gq+8, same cols)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = nt * 8 + 2 * tq;
                const int r0 = rbase + gq, r1 = rbase + gq + 8;
                if (r0 < N) {
                    part[((long long)ks * N + r0) * RP + col] = acc[nt][0];
                    part[((long long)ks * N + r0) * RP + col + 1] = acc[nt][1];
                }
                if (r1 < N) {
                    part[((long long)ks * N + r1) * RP + col] = acc[nt][2];
                    part[((long long)ks * N + r1) * RP + col + 1] = acc[nt][3];
                }
            }
        }
    } else {
        // fp32 engine (fp32 weights): one row at a time, lanes split K
        const float *xf = reinterpret_cast<const float *>(xs);
        for (int rr = 0; rr < 16; ++rr) {
            const int row = rbase + rr;
            if (row >= N) break;
            const T *w = sk_row<T, SE>(P, layer, row, K) + k0;
            float acc[RP];
#pragma unroll
            for (int r = 0; r < RP; ++r) acc[r] = 0.f;
            for (int k = lane; k < kseg; k += 32) {
                const float wv = (float)w[k];
#pragma unroll
                for (int r = 0; r < RP; ++r) acc[r] = fmaf(wv, xf[r * pitch + k], acc[r]);
            }
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const float s = warp_sum(acc[r]);
                if (lane == 0) part[((long long)ks * N + row) * RP + r] = s;
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(P->sk_cnt + rb, 1) == nks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- epilogue for rows [rb*128, rb*128+128): sum the K-split partials in split order.
    // Each thread owns items tid, tid+256, ...; the loads of 4 items x 8 splits are issued
    // before any add, so the chain costs a few L2 round trips, not nks of them.
    const int rlo = rb * SK_ROWS, rhi = min(N, rlo + SK_ROWS);
    const int d = P->d;
    float *ys = reinterpret_cast<float *>(sk_smem);   // [128][RP] (reuses the x buffer)
    __syncthreads();
    const int nitems = (rhi - rlo) * R;
    for (int i0 = threadIdx.x; i0 < nitems; i0 += 4 * blockDim.x) {
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
        long long base[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = min(i0 + e * (int)blockDim.x, nitems - 1);
            const int rl = idx / R, r = idx - rl * R;
            base[e] = (long long)(rlo + rl) * RP + r;
        }
        for (int q0 = 0; q0 < nks; q0 += 8) {
            float v[4][8];
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    v[e][u] = (i0 + e * (int)blockDim.x < nitems && q0 + u < nks)
                                  ? __ldcg(part + (long long)(q0 + u) * N * RP + base[e]) : 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (q0 + u < nks) sum[e] += v[e][u];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = i0 + e * blockDim.x;
            if (idx >= nitems) continue;
            const int rl = idx / R, r = idx - rl * R;
            const int row = rlo + rl;
            if (SE == SE_PROJ) P->Xp[(long long)r * d + row] = sum[e];
            else if (SE == SE_OPROJ || SE == SE_DOWN) P->Xp[(long long)r * d + row] += sum[e];
            else if (SE == SE_GATEUP) P->GUp[(long long)r * 2 * P->F + row] = sum[e];
            else ys[rl * RP + r] = sum[e];
        }
    }
    if (SE == SE_QKV) {
        __syncthreads();
        const int hd = P->hd, half = hd / 2, Hkv = P->Hkv;
        const long long rowstride = (long long)Hkv * hd;
        T *kc = reinterpret_cast<T *>(P->pkc) + (long long)layer * P->kv_stride;
        T *vc = reinterpret_cast<T *>(P->pvc) + (long long)layer * P->kv_stride;
        for (int idx = threadIdx.x; idx < (rhi - rlo) * R; idx += blockDim.x) {
            const int rl = idx / R, r = idx - rl * R;
            const int row = rlo + rl;
            const int pos = pr.pos0 + r;
            const int i = row % hd;
            if (row < P->q_rows + P->kv_rows) {
                // q or k: rotate-half RoPE at the row's position
                const int ii = i < half ? i : i - half;
                const float2 cs = P->rope[(long long)pos * half + ii];
                const float a = ys[(rl - i + ii) * RP + r], b = ys[(rl - i + ii + half) * RP + r];
                const float v = i < half ? a * cs.x - b * cs.y : b * cs.x + a * cs.y;
                if (row < P->q_rows)
                    P->QKVp[(long long)r * P->qkv_rows + row] = v;
                else {
                    const int kr = row - P->q_rows;
                    kc[(long long)pos * rowstride + kr] = WTraits<T>::store(v);
                }
            } else {
                const int vr = row - P->q_rows - P->kv_rows;
                vc[(long long)pos * rowstride + vr] = WTraits<T>::store(ys[rl * RP + r]);
            }
        }
    }
    if (threadIdx.x == 0) P->sk_cnt[rb] = 0;
    if (SE == SE_PROJ || SE == SE_OPROJ || SE == SE_DOWN) {
        // last block overall: RMS statistics of the updated rows for the next norm
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_glast = atomicAdd(P->sk_cnt + nrb, 1) == nrb - 1;
        __syncthreads();
        if (!s_glast) return;
        __threadfence();
        // all rows at once: per-thread sums of squares with the rows' loads in flight
        // together, then one fixed-order reduction over warps per row
        float ss[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) ss[r] = 0.f;
        for (int k = threadIdx.x; k < d; k += blockDim.x) {
#pragma unroll
            for (int r = 0; r < RP; ++r)
                if (r < R) {
                    const float v = __ldcg(P->Xp + (long long)r * d + k);
                    ss[r] = fmaf(v, v, ss[r]);
                }
        }
        float *wred = reinterpret_cast<float *>(sk_smem);   // [8 warps][RP]
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const float t = warp_sum(ss[r]);
            if (lane == 0) wred[warp * RP + r] = t;
        }
        __syncthreads();
        if (threadIdx.x < R) {
            float t = 0.f;
            for (int w = 0; w < SK_THREADS / 32; ++w) t += wred[w * RP + threadIdx.x];
            P->inv_rms_p[threadIdx.x] = 1.0f / sqrtf(t / (float)d + P->eps);
        }
        if (threadIdx.x == 0) P->sk_cnt[nrb] = 0;
    }
}

// ---------------------------------------------------------------------------------
static int sk_smem_for(const Plan &h, int K, int nks, int NT, int xbytes) {
    const int nch = K / SK_KCHUNK;
    const int kmax = ((nch + nks - 1) / nks) * SK_KCHUNK;
    const int pitch = kmax + (xbytes == 2 ? 32 : 4);
    int b = NT * 8 * pitch * xbytes;
    const int ys = SK_ROWS * NT * 8 * 4;
    return b > ys ? b : ys;
}

void sk_plan(const Plan &h, int num_sms, SkPlan &sk) {
    const int Ns[5] = {h.d, h.qkv_rows, h.d, 2 * h.F, h.d};
    const int Ks[5] = {h.nB * h.d, h.d, h.q_rows, h.d, h.F};
    sk.NT = (h.n + 1 + 7) / 8;
    const int xbytes = h.dtype == SPD_BF16 ? 2 : 4;
    sk.smem = 0;
    for (int i = 0; i < 5; ++i) {
        const int nrb = (Ns[i] + SK_ROWS - 1) / SK_ROWS;
        const int nch = Ks[i] / SK_KCHUNK;
        int nks = (2 * num_sms + nrb - 1) / nrb;
        if (nks < 1) nks = 1;
        if (nks > nch) nks = nch;
        sk.nks[i] = nks;
        const int sm = sk_smem_for(h, Ks[i], nks, sk.NT, xbytes);
        if (sm > sk.smem) sk.smem = sm;
    }
}

template <typename T, int NT, int XM, int SE>
static void sk_launch(const Plan *P, int layer, int N, int K, int nks, int smem, cudaStream_t s) {
    const int nrb = (N + SK_ROWS - 1) / SK_ROWS;
    k_skinny<T, NT, XM, SE><<<nrb * nks, SK_THREADS, smem, s>>>(P, layer, N, K, nks);
}

template <typename T, int NT>
static void pdm_step_nt(const Plan *P, const Plan &h, const SkPlan &sk, cudaStream_t s) {
    sk_launch<T, NT, XM_FEAT, SE_PROJ>(P, 0, h.d, h.nB * h.d, sk.nks[0], sk.smem, s);
    for (int li = 0; li < h.Ls; ++li) {
        sk_launch<T, NT, XM_NORM1, SE_QKV>(P, li, h.qkv_rows, h.d, sk.nks[1], sk.smem, s);
        launch_pdm_attn<T>(P, h, li, s);
        sk_launch<T, NT, XM_ATT, SE_OPROJ>(P, li, h.d, h.q_rows, sk.nks[2], sk.smem, s);
        sk_launch<T, NT, XM_NORM2, SE_GATEUP>(P, li, 2 * h.F, h.d, sk.nks[3], sk.smem, s);
        sk_launch<T, NT, XM_SILU, SE_DOWN>(P, li, h.d, h.F, sk.nks[4], sk.smem, s);
    }
}

template <typename T>
void launch_pdm_step(const Plan *P, const Plan &h, const SkPlan &sk, cudaStream_t s) {
    switch (sk.NT) {
        case 1: pdm_step_nt<T, 1>(P, h, sk, s); break;
        case 2: pdm_step_nt<T, 2>(P, h, sk, s); break;
        case 3: pdm_step_nt<T, 3>(P, h, sk, s); break;
        default: pdm_step_nt<T, 4>(P, h, sk, s); break;
    }
}

template <typename T, int NT>
static void set_attr_nt(int smem) {
    cudaFuncSetAttribute(k_skinny<T, NT, XM_FEAT, SE_PROJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_skinny<T, NT, XM_NORM1, SE_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_skinny<T, NT, XM_ATT, SE_OPROJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_skinny<T, NT, XM_NORM2, SE_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_skinny<T, NT, XM_SILU, SE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

void set_pdm_attributes(int smem) {
    set_attr_nt<float, 1>(smem);
    set_attr_nt<float, 2>(smem);
    set_attr_nt<float, 3>(smem);
    set_attr_nt<float, 4>(smem);
    set_attr_nt<__nv_bfloat16, 1>(smem);
    set_attr_nt<__nv_bfloat16, 2>(smem);
    set_attr_nt<__nv_bfloat16, 3>(smem);
    set_attr_nt<__nv_bfloat16, 4>(smem);
}

template void launch_pdm_step<float>(const Plan *, const Plan &, const SkPlan &, cudaStream_t);
template void launch_pdm_step<__nv_bfloat16>(const Plan *, const Plan &, const SkPlan &, cudaStream_t);

}  // namespace spd
