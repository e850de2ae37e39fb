// Prefill: the prompt's dense pass through all target layers, the draft module's cached
// prefix, and the first token.  Not part of the timed step; it fills what the step
// needs: every layer's K,V for the prompt positions and the draft module's K,V built
// from full-depth anchor features of the verified prefix (machine review, "What carries
// the argument": verified positions use every anchor depth).
//
// The prompt is processed in chunks of pf_rows positions (each chunk attends causally to
// the cache of the chunks before it).  bf16 weights: every projection is a tensor-core
// GEMM (umma.cuh: tcgen05, TMEM accumulators, TMA-fed operands) whose activation operand
// comes as two bf16 parts written by the kernel before it (the norm, the attention
// output's split, SiLU(gate) * up, the anchors' split), and the causal attention runs on
// tensor cores too (mma.sync, flash-attention order, the fp32 K/V rows split into fp16 parts).  fp32
// weights: an fp32 tiled CUDA-core GEMM and attention.
#include <cudaTypedefs.h>

#include <string>

#include "umma.cuh"

namespace spd {

// ---------------------------------------------------------------------------------
// C[M][N] (+)= A[M][K] * W[N][K]^T ; 128x128 tiles, 8x8 outputs per thread
constexpr int GM = 128, GN = 128, GK = 8;

template <typename T>
__global__ void __launch_bounds__(256) k_pf_gemm(const float *__restrict__ A, int lda, const T *__restrict__ W, int N,
                                                int K, float *__restrict__ C, int ldc, int M, int accumulate) {
    __shared__ __align__(16) float As[GK][GM + 4];
    __shared__ __align__(16) float Ws[GK][GN + 4];
    const int t = threadIdx.x;
    const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
    const int ty = t / 16, tx = t % 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    const int lr = t / 2, lk = (t % 2) * 4;
    for (int k0 = 0; k0 < K; k0 += GK) {
        {
            const int m = m0 + lr;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < M) v = *reinterpret_cast<const float4 *>(A + (long long)m * lda + k0 + lk);
            As[lk + 0][lr] = v.x;
            As[lk + 1][lr] = v.y;
            As[lk + 2][lr] = v.z;
            As[lk + 3][lr] = v.w;
            const int n = n0 + lr;
            float w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;
            if (n < N) {
                const T *wp = W + (long long)n * K + k0 + lk;
                w0 = WTraits<T>::get(wp, 0);
                w1 = WTraits<T>::get(wp, 1);
                w2 = WTraits<T>::get(wp, 2);
                w3 = WTraits<T>::get(wp, 3);
            }
            Ws[lk + 0][lr] = w0;
            Ws[lk + 1][lr] = w1;
            Ws[lk + 2][lr] = w2;
            Ws[lk + 3][lr] = w3;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < GK; ++k) {
            float a[8], w[8];
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Ws[k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Ws[k][64 + tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            w[0] = b0.x; w[1] = b0.y; w[2] = b0.z; w[3] = b0.w;
            w[4] = b1.x; w[5] = b1.y; w[6] = b1.z; w[7] = b1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
            if (n >= N) continue;
            float *c = C + (long long)m * ldc + n;
            *c = accumulate ? *c + acc[i][j] : acc[i][j];
        }
    }
}

template <typename T>
static void pf_gemm(const float *A, int lda, const void *W, int N, int K, float *C, int ldc, int M, int acc,
                    cudaStream_t s) {
    dim3 grid((N + GN - 1) / GN, (M + GM - 1) / GM);
    k_pf_gemm<T><<<grid, 256, 0, s>>>(A, lda, reinterpret_cast<const T *>(W), N, K, C, ldc, M, acc);
}

// ---------------------------------------------------------------------------------
template <typename T>
__global__ void k_pf_embed(const Plan *__restrict__ P, const int *__restrict__ prompt, int p0) {
    const int m = blockIdx.x, d = P->d;
    int tok = prompt[p0 + m];
    if (tok < 0 || tok >= P->V) {
        if (threadIdx.x == 0) P->st->error = ERR_TOKEN;
        tok = 0;
    }
    const T *e = reinterpret_cast<const T *>(P->embed) + (long long)tok * d;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float v = WTraits<T>::get(e, k);
        P->pf_H[(long long)m * d + k] = v;
        P->pf_ANCH[(long long)m * P->nB * d + k] = v;
    }
}

__global__ void k_pf_norm(const float *__restrict__ src, float *__restrict__ dst, const float *__restrict__ g, int d,
                          float eps) {
    __shared__ float red[40];
    const float *x = src + (long long)blockIdx.x * d;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) ss = fmaf(x[k], x[k], ss);
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int k = threadIdx.x; k < d; k += blockDim.x) dst[(long long)blockIdx.x * d + k] = (x[k] * inv) * g[k];
}

template <typename T>
__global__ void k_pf_rope_kv(const Plan *__restrict__ P, float *__restrict__ qkv, int p0, T *__restrict__ kc,
                             T *__restrict__ vc) {
    const int m = blockIdx.x, pos = p0 + m;
    const int hd = P->hd, half = hd / 2;
    float *row = qkv + (long long)m * P->qkv_rows;
    const float2 *cs = P->rope + (long long)pos * half;
    const long long rs = (long long)P->Hkv * hd;
    // q heads (in place)
    for (int idx = threadIdx.x; idx < P->Hq * half; idx += blockDim.x) {
        const int h = idx / half, i = idx % half;
        float *q = row + (long long)h * hd;
        const float a = q[i], b = q[i + half];
        const float2 r = cs[i];
        q[i] = a * r.x - b * r.y;
        q[i + half] = b * r.x + a * r.y;
    }
    for (int idx = threadIdx.x; idx < P->Hkv * half; idx += blockDim.x) {
        const int h = idx / half, i = idx % half;
        const float *k = row + P->q_rows + (long long)h * hd;
        const float a = k[i], b = k[i + half];
        const float2 r = cs[i];
        kc[(long long)pos * rs + (long long)h * hd + i] = WTraits<T>::store(a * r.x - b * r.y);
        kc[(long long)pos * rs + (long long)h * hd + i + half] = WTraits<T>::store(b * r.x + a * r.y);
    }
    for (int idx = threadIdx.x; idx < P->kv_rows; idx += blockDim.x)
        vc[(long long)pos * rs + idx] = WTraits<T>::store(row[P->q_rows + P->kv_rows + idx]);
}

// Causal attention of M prompt rows (positions p0..p0+M-1) over cache positions
// 0..p0+M-1.  CTA = (block of QB query rows, kv head); thread = (row, head of the GQA
// group, quarter of the head dim; dims sub, sub+4, ...).  Online softmax over 64-key
// tiles staged in shared memory.
constexpr int PF_KT = 64;
template <typename T, int HD>
__global__ void __launch_bounds__(256) k_pf_attn(const Plan *__restrict__ P, const float *__restrict__ qkv, int p0,
                                                 int M, const T *__restrict__ kc, const T *__restrict__ vc,
                                                 float *__restrict__ out) {
    extern __shared__ __align__(16) float kvs[];
    constexpr int hd = HD, DS = HD / 4;
    const int G = P->Hq / P->Hkv, Hkv = P->Hkv;
    const int QB = 64 / G;
    const int g = blockIdx.y;
    const int t = threadIdx.x;
    const int qi = t / (G * 4), h = (t / 4) % G, sub = t % 4;
    const int m = blockIdx.x * QB + qi;
    const bool live = m < M;
    const int qpos = p0 + (live ? m : M - 1);
    float q[DS], o[DS];
    const float *qp = qkv + (long long)(live ? m : M - 1) * P->qkv_rows + (long long)(g * G + h) * hd;
#pragma unroll
    for (int e = 0; e < DS; ++e) {
        q[e] = qp[sub + 4 * e] * P->scale;
        o[e] = 0.f;
    }
    float mx = -INFINITY, l = 0.f;
    const int last_row = min(M, (blockIdx.x + 1) * QB) - 1;
    const int kend = p0 + last_row + 1;
    float *Ks = kvs, *Vs = kvs + PF_KT * hd;
    const long long rs = (long long)Hkv * hd;
    for (int kt0 = 0; kt0 < kend; kt0 += PF_KT) {
        __syncthreads();
        for (int idx = t; idx < PF_KT * hd; idx += blockDim.x) {
            const int j = idx / hd, e = idx % hd;
            const int kp = kt0 + j;
            float kv = 0.f, vv = 0.f;
            if (kp < kend) {
                kv = WTraits<T>::get(kc, (long long)kp * rs + (long long)g * hd + e);
                vv = WTraits<T>::get(vc, (long long)kp * rs + (long long)g * hd + e);
            }
            Ks[idx] = kv;
            Vs[idx] = vv;
        }
        __syncthreads();
        const int jn = min(PF_KT, kend - kt0);
        for (int j = 0; j < jn; ++j) {
            float s = 0.f;
            const float *kr = Ks + j * hd + sub;
#pragma unroll
            for (int e = 0; e < DS; ++e) s = fmaf(q[e], kr[4 * e], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (kt0 + j <= qpos) {
                if (s > mx) {
                    const float corr = expf(mx - s);
                    l *= corr;
#pragma unroll
                    for (int e = 0; e < DS; ++e) o[e] *= corr;
                    mx = s;
                }
                const float p = expf(s - mx);
                l += p;
                const float *vr = Vs + j * hd + sub;
#pragma unroll
                for (int e = 0; e < DS; ++e) o[e] = fmaf(p, vr[4 * e], o[e]);
            }
        }
    }
    if (live) {
        float *op = out + (long long)m * P->q_rows + (long long)(g * G + h) * hd;
#pragma unroll
        for (int e = 0; e < DS; ++e) op[sub + 4 * e] = o[e] / l;
    }
}

// ---- causal attention of a prompt chunk on tensor cores (fp32 K/V cache) ------------------
// CTA = 64 query rows of one query head (4 warps x 16 rows), flash-attention order over key
// tiles of 32 positions.  cp.async copies the next tile's fp32 K and V rows into a staging
// buffer while the warps work on the current tile, which has been split into fp16 parts
// hi = fp16(x) and lo = fp16(x - hi) (about 21 bits of each value).  Scores S = Q K^T by
// mma.sync m16n8k16 as q_hi k_hi + q_lo k_hi + q_hi k_lo (q pre-scaled by 1/sqrt(hd) and split
// the same way; the lo x lo term lies below the fp32 accumulation's resolution), an online
// softmax per row in registers, the probabilities split the same way and
// O += P_hi V_hi + P_lo V_hi + P_hi V_lo; the causal mask applies on the diagonal tile only.
// Output fp32 [row][Hq * hd], as the tensor-core O projection's input split expects.
constexpr int FA_BQ = 64, FA_BK = 32, FA_THREADS = 128;   // 32-key tiles: two CTAs per SM
template <int HD> __host__ __device__ constexpr int fa_pitch() { return HD + 8; }   // halfs; ldmatrix rows on distinct banks
template <int HD> __host__ __device__ constexpr int fa_smem_bytes() {
    // q hi / lo, K hi / lo, V hi / lo (fp16 tiles), then the fp32 K and V staging rows
    return (2 * FA_BQ + 4 * FA_BK) * fa_pitch<HD>() * 2 + 2 * FA_BK * HD * 4;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// fp16 parts of four fp32 values: hi = fp16(x) (range-clamped), lo = fp16(x - hi)
__device__ __forceinline__ void split_h4(const float4 v, __half *hi, __half *lo) {
    const float x[4] = {v.x, v.y, v.z, v.w};
    __half h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = __float2half_rn(fminf(fmaxf(x[i], -F16_MAX), F16_MAX));
        l[i] = __float2half_rn(x[i] - __half2float(h[i]));
    }
    *reinterpret_cast<uint2 *>(hi) = make_uint2((uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16),
                                                (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16));
    *reinterpret_cast<uint2 *>(lo) = make_uint2((uint32_t)__half_as_ushort(l[0]) | ((uint32_t)__half_as_ushort(l[1]) << 16),
                                                (uint32_t)__half_as_ushort(l[2]) | ((uint32_t)__half_as_ushort(l[3]) << 16));
}

template <int HD>
__global__ void __launch_bounds__(FA_THREADS) k_pf_fa(const Plan *__restrict__ P, const float *__restrict__ qkv, int p0,
                                                      int M, const float *__restrict__ kc, const float *__restrict__ vc,
                                                      float *__restrict__ out) {
    extern __shared__ __align__(16) unsigned char fa_raw[];
    constexpr int PT = fa_pitch<HD>(), NT = FA_BK / 8, KS = HD / 16, NO = HD / 8;
    __half *Qh = reinterpret_cast<__half *>(fa_raw), *Ql = Qh + FA_BQ * PT;
    __half *Kh = Ql + FA_BQ * PT, *Kl = Kh + FA_BK * PT, *Vh = Kl + FA_BK * PT, *Vl = Vh + FA_BK * PT;
    float *Kf = reinterpret_cast<float *>(Vl + FA_BK * PT), *Vf = Kf + FA_BK * HD;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int h = blockIdx.y, G = P->Hq / P->Hkv, g = h / G;
    const int q0 = blockIdx.x * FA_BQ;
    const long long rs = (long long)P->Hkv * HD;
    const int kv_end = p0 + M;                                  // keys written so far
    const int kend = min(kv_end, p0 + q0 + FA_BQ);              // keys any row of this CTA sees
    const int ntiles = (kend + FA_BK - 1) / FA_BK;
    const float scale = P->scale;
    // ---- fp32 K / V rows of tile t into the staging rows (rows past the written keys are zero)
    auto stage_tile = [&](int t) {
        const int k0 = t * FA_BK;
        for (int c = tid; c < FA_BK * HD / 4; c += FA_THREADS) {
            const int j = c / (HD / 4), e = (c - j * (HD / 4)) * 4;
            float *kd = Kf + j * HD + e, *vd = Vf + j * HD + e;
            if (k0 + j < kv_end) {
                cp_async16(kd, kc + (long long)(k0 + j) * rs + (long long)g * HD + e);
                cp_async16(vd, vc + (long long)(k0 + j) * rs + (long long)g * HD + e);
            } else {
                *reinterpret_cast<float4 *>(kd) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(vd) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // ---- the staged rows as fp16 hi / lo tiles (after every thread's copies have landed)
    auto split_tile = [&]() {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        for (int c = tid; c < FA_BK * HD / 4; c += FA_THREADS) {
            const int j = c / (HD / 4), e = (c - j * (HD / 4)) * 4;
            split_h4(*reinterpret_cast<const float4 *>(Kf + j * HD + e), Kh + j * PT + e, Kl + j * PT + e);
            split_h4(*reinterpret_cast<const float4 *>(Vf + j * HD + e), Vh + j * PT + e, Vl + j * PT + e);
        }
        __syncthreads();
    };
    stage_tile(0);
    // ---- q (rotated already), pre-scaled by 1/sqrt(hd), as fp16 hi + lo
    for (int c = tid; c < FA_BQ * HD; c += FA_THREADS) {
        const int r = c / HD, e = c - r * HD;
        const int m = min(q0 + r, M - 1);
        const float v = qkv[(long long)m * P->qkv_rows + (long long)h * HD + e] * scale;
        const __half hi = __float2half_rn(v);
        Qh[r * PT + e] = hi;
        Ql[r * PT + e] = __float2half_rn(v - __half2float(hi));
    }
    split_tile();
    float o[NO][4];
#pragma unroll
    for (int i = 0; i < NO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int r0 = warp * 16;                                   // this warp's first row in the tile
    const int qpos0 = p0 + q0 + r0 + gq, qpos1 = qpos0 + 8;      // positions of the thread's two rows
    const uint32_t qh_addr = smem_u32(Qh + (r0 + (lane & 15)) * PT + (lane >> 4) * 8);
    const uint32_t ql_addr = smem_u32(Ql + (r0 + (lane & 15)) * PT + (lane >> 4) * 8);
    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) stage_tile(t + 1);   // the staging rows are free once split
        // ---- S = Q K^T: 16 rows x 64 keys per warp
        float sc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3;
            ldsm_x4(qh_addr + ks * 32, ah0, ah1, ah2, ah3);
            ldsm_x4(ql_addr + ks * 32, al0, al1, al2, al3);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                // keys 16 np .. 16 np + 15: two n8 tiles, hi and lo parts
                uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
                const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int off = key * PT + ks * 16 + ((lane >> 3) & 1) * 8;
                ldsm_x4(smem_u32(Kh + off), b0, b1, b2, b3);
                ldsm_x4(smem_u32(Kl + off), c0, c1, c2, c3);
                mma_f16(sc[2 * np], ah0, ah1, ah2, ah3, b0, b1);
                mma_f16(sc[2 * np], al0, al1, al2, al3, b0, b1);
                mma_f16(sc[2 * np], ah0, ah1, ah2, ah3, c0, c1);
                mma_f16(sc[2 * np + 1], ah0, ah1, ah2, ah3, b2, b3);
                mma_f16(sc[2 * np + 1], al0, al1, al2, al3, b2, b3);
                mma_f16(sc[2 * np + 1], ah0, ah1, ah2, ah3, c2, c3);
            }
        }
        // ---- causal mask on the diagonal tile, online softmax
        const int k0 = t * FA_BK;
        if (k0 + FA_BK - 1 > qpos0) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int key = k0 + i * 8 + 2 * tq;
                if (key > qpos0) sc[i][0] = -INFINITY;
                if (key + 1 > qpos0) sc[i][1] = -INFINITY;
                if (key > qpos1) sc[i][2] = -INFINITY;
                if (key + 1 > qpos1) sc[i][3] = -INFINITY;
            }
        }
        float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            mx[0] = fmaxf(mx[0], fmaxf(sc[i][0], sc[i][1]));
            mx[1] = fmaxf(mx[1], fmaxf(sc[i][2], sc[i][3]));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float corr[2], ls[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) corr[r] = mx[r] == -INFINITY ? 1.f : expf(mrow[r] - mx[r]);
        uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const float e0 = mx[0] == -INFINITY ? 0.f : expf(sc[i][0] - mx[0]);
            const float e1 = mx[0] == -INFINITY ? 0.f : expf(sc[i][1] - mx[0]);
            const float e2 = mx[1] == -INFINITY ? 0.f : expf(sc[i][2] - mx[1]);
            const float e3 = mx[1] == -INFINITY ? 0.f : expf(sc[i][3] - mx[1]);
            ls[0] += e0 + e1;
            ls[1] += e2 + e3;
            const __half2 h01 = __floats2half2_rn(e0, e1), h23 = __floats2half2_rn(e2, e3);
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            ph[i][0] = *reinterpret_cast<const uint32_t *>(&h01);
            ph[i][1] = *reinterpret_cast<const uint32_t *>(&h23);
            pl[i][0] = pack_h2(e0 - f01.x, e1 - f01.y);
            pl[i][1] = pack_h2(e2 - f23.x, e3 - f23.y);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 1);
            ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 2);
            lrow[r] = lrow[r] * corr[r] + ls[r];
            mrow[r] = mx[r];
        }
#pragma unroll
        for (int i = 0; i < NO; ++i) {
            o[i][0] *= corr[0];
            o[i][1] *= corr[0];
            o[i][2] *= corr[1];
            o[i][3] *= corr[1];
        }
        // ---- O += P V
#pragma unroll
        for (int s = 0; s < FA_BK / 16; ++s) {
            const uint32_t a0 = ph[2 * s][0], a1 = ph[2 * s][1], a2 = ph[2 * s + 1][0], a3 = ph[2 * s + 1][1];
            const uint32_t l0 = pl[2 * s][0], l1 = pl[2 * s][1], l2 = pl[2 * s + 1][0], l3 = pl[2 * s + 1][1];
#pragma unroll
            for (int np = 0; np < NO / 2; ++np) {
                uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
                const int key = s * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int off = key * PT + np * 16 + (lane >> 4) * 8;
                ldsm_x4_t(smem_u32(Vh + off), b0, b1, b2, b3);
                ldsm_x4_t(smem_u32(Vl + off), c0, c1, c2, c3);
                mma_f16(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_f16(o[2 * np], l0, l1, l2, l3, b0, b1);
                mma_f16(o[2 * np], a0, a1, a2, a3, c0, c1);
                mma_f16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
                mma_f16(o[2 * np + 1], l0, l1, l2, l3, b2, b3);
                mma_f16(o[2 * np + 1], a0, a1, a2, a3, c2, c3);
            }
        }
        __syncthreads();   // every warp is done with this tile's parts
        if (t + 1 < ntiles) split_tile();
    }
    // ---- normalise and store the warp's rows
    const int m_a = q0 + r0 + gq, m_b = m_a + 8;
    const float inv0 = 1.0f / lrow[0], inv1 = 1.0f / lrow[1];
#pragma unroll
    for (int i = 0; i < NO; ++i) {
        const int e = i * 8 + 2 * tq;
        if (m_a < M) *reinterpret_cast<float2 *>(out + (long long)m_a * P->q_rows + (long long)h * HD + e) =
                         make_float2(o[i][0] * inv0, o[i][1] * inv0);
        if (m_b < M) *reinterpret_cast<float2 *>(out + (long long)m_b * P->q_rows + (long long)h * HD + e) =
                         make_float2(o[i][2] * inv1, o[i][3] * inv1);
    }
}

// ---- the tensor-core GEMMs' activation operand: two bf16 parts per value ------------------
__device__ __forceinline__ void split_store(__nv_bfloat16 *A2, long long lo_off, long long i, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    A2[i] = hi;
    A2[lo_off + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// rms(x) * g of every row, written as the hi / lo parts of A2 (row pitch d)
__global__ void k_pf_norm_split(const float *__restrict__ src, __nv_bfloat16 *__restrict__ A2, int rows_cap,
                                const float *__restrict__ g, int d, float eps) {
    __shared__ float red[40];
    const float *x = src + (long long)blockIdx.x * d;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) ss = fmaf(x[k], x[k], ss);
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    const long long lo = (long long)rows_cap * d;
    for (int k = threadIdx.x; k < d; k += blockDim.x)
        split_store(A2, lo, (long long)blockIdx.x * d + k, (x[k] * inv) * g[k]);
}

// rows of src (pitch ld, K values each) as the hi / lo parts of A2 (row pitch K)
__global__ void k_pf_split(const float *__restrict__ src, int ld, int K, int M, __nv_bfloat16 *__restrict__ A2,
                           int rows_cap) {
    const long long total = (long long)M * K, lo = (long long)rows_cap * K;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / K, k = i - m * K;
        split_store(A2, lo, i, src[m * ld + k]);
    }
}

// SiLU(gate) * up of every row as the hi / lo parts of A2 (row pitch F)
__global__ void k_pf_silu_split(const Plan *__restrict__ P, int M) {
    const int F = P->F;
    const long long total = (long long)M * F, lo = (long long)P->pf_rows * F;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / F, k = i - m * F;
        split_store(P->pf_A2, lo, i, silu_f(P->pf_GU[m * 2 * F + k]) * P->pf_GU[m * 2 * F + F + k]);
    }
}

__global__ void k_pf_silu(const Plan *__restrict__ P, int M) {
    const int F = P->F;
    const long long total = (long long)M * F;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / F, k = i - m * F;
        P->pf_XN[i] = silu_f(P->pf_GU[m * 2 * F + k]) * P->pf_GU[m * 2 * F + F + k];
    }
}

__global__ void k_pf_anchor(const Plan *__restrict__ P, int M, int a) {
    const int d = P->d;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)M * d;
         i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / d, k = i - m * d;
        P->pf_ANCH[(m * P->nB + a) * d + k] = P->pf_H[i];
    }
}

// logits of one row: pf_logits[v] = W_lm[v] . (rms(h) * g_f)
template <typename T>
__global__ void __launch_bounds__(256) k_pf_logits(const Plan *__restrict__ P, const float *__restrict__ h) {
    extern __shared__ __align__(16) float xs[];
    __shared__ float red[40];
    const int d = P->d, V = P->V;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) ss = fmaf(h[k], h[k], ss);
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + P->eps);
    for (int k = threadIdx.x; k < d; k += blockDim.x) xs[k] = (h[k] * inv) * P->gf[k];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T *W = reinterpret_cast<const T *>(P->lm_head);
    for (int v = blockIdx.x * 8 + warp; v < V; v += gridDim.x * 8) {
        float acc = 0.f;
        for (int k = lane; k < d; k += 32) acc = fmaf(WTraits<T>::get(W, (long long)v * d + k), xs[k], acc);
        acc = warp_sum(acc);
        if (lane == 0) P->pf_logits[v] = acc;
    }
}

// ---------------------------------------------------------------------------------
// Tensor-core GEMM launch (bf16 weights): C[M][N] (+)= (A_hi + A_lo)[M][K] . W[N][K]^T with
// A in pf_A2 (row pitch K).  The tensor maps are encoded on the host per call (a few
// microseconds); the tile width BN is the largest of 256 / 128 / 64 that divides N and
// still gives about one CTA per SM.
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 map over rows x K (K contiguous), box 64 (K) x box_rows, 128-byte swizzle
static bool tmap_bf16(CUtensorMap *m, const void *base, int K, long long rows, int box_rows) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)UM_BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int g_num_sms = 0;

template <int BN>
static bool um_launch(const Plan &h, const void *W, int N, int K, float *C, int ldc, int M, int acc, cudaStream_t s) {
    CUtensorMap ta, tw;
    if (!tmap_bf16(&ta, h.pf_A2, K, 2LL * h.pf_rows, UM_BM) || !tmap_bf16(&tw, W, K, N, BN)) return false;
    const UmmaArgs a{C, ldc, M, N, K, h.pf_rows, acc, &h.st->error};
    k_umma_gemm<BN><<<dim3(N / BN, (M + UM_BM - 1) / UM_BM), UM_THREADS, UM_SMEM, s>>>(ta, tw, a);
    return true;
}

static bool um_gemm(const Plan &h, const void *W, int N, int K, float *C, int ldc, int M, int acc, cudaStream_t s) {
    const int mt = (M + UM_BM - 1) / UM_BM, want = g_num_sms > 0 ? g_num_sms : 148;
    if (N % 256 == 0 && (N / 256) * mt >= want) return um_launch<256>(h, W, N, K, C, ldc, M, acc, s);
    if (N % 128 == 0 && ((N / 128) * mt >= want || N % 64 != 0)) return um_launch<128>(h, W, N, K, C, ldc, M, acc, s);
    return um_launch<64>(h, W, N, K, C, ldc, M, acc, s);
}

template <typename T>
static bool pf_layer(const Plan *P, const Plan &h, const LayerW &w, KvT<T> *kc, KvT<T> *vc, float *H, int p0, int M,
                     cudaStream_t s) {
    using KV = KvT<T>;
    constexpr bool TC = sizeof(T) == 2;   // bf16 weights: tensor-core GEMMs
    const int d = h.d;
    bool ok = true;
    if (TC) {
        k_pf_norm_split<<<M, 256, 0, s>>>(H, h.pf_A2, h.pf_rows, w.g1, d, h.eps);
        ok = ok && um_gemm(h, w.wq, h.q_rows, d, h.pf_QKV, h.qkv_rows, M, 0, s);
        ok = ok && um_gemm(h, w.wk, h.kv_rows, d, h.pf_QKV + h.q_rows, h.qkv_rows, M, 0, s);
        ok = ok && um_gemm(h, w.wv, h.kv_rows, d, h.pf_QKV + h.q_rows + h.kv_rows, h.qkv_rows, M, 0, s);
    } else {
        k_pf_norm<<<M, 256, 0, s>>>(H, h.pf_XN, w.g1, d, h.eps);
        pf_gemm<T>(h.pf_XN, d, w.wq, h.q_rows, d, h.pf_QKV, h.qkv_rows, M, 0, s);
        pf_gemm<T>(h.pf_XN, d, w.wk, h.kv_rows, d, h.pf_QKV + h.q_rows, h.qkv_rows, M, 0, s);
        pf_gemm<T>(h.pf_XN, d, w.wv, h.kv_rows, d, h.pf_QKV + h.q_rows + h.kv_rows, h.qkv_rows, M, 0, s);
    }
    k_pf_rope_kv<KV><<<M, 256, 0, s>>>(P, h.pf_QKV, p0, kc, vc);
    if constexpr (TC) {
        const dim3 fg((M + FA_BQ - 1) / FA_BQ, h.Hq);
        if (h.hd == 128) k_pf_fa<128><<<fg, FA_THREADS, fa_smem_bytes<128>(), s>>>(P, h.pf_QKV, p0, M, kc, vc, h.pf_ATT);
        else k_pf_fa<64><<<fg, FA_THREADS, fa_smem_bytes<64>(), s>>>(P, h.pf_QKV, p0, M, kc, vc, h.pf_ATT);
    } else {
        const int G = h.Hq / h.Hkv, QB = 64 / G;
        dim3 ag((M + QB - 1) / QB, h.Hkv);
        const size_t sm = 2 * PF_KT * h.hd * sizeof(float);
        if (h.hd == 128) k_pf_attn<KV, 128><<<ag, 256, sm, s>>>(P, h.pf_QKV, p0, M, kc, vc, h.pf_ATT);
        else k_pf_attn<KV, 64><<<ag, 256, sm, s>>>(P, h.pf_QKV, p0, M, kc, vc, h.pf_ATT);
    }
    if (TC) {
        k_pf_split<<<1024, 256, 0, s>>>(h.pf_ATT, h.q_rows, h.q_rows, M, h.pf_A2, h.pf_rows);
        ok = ok && um_gemm(h, w.wo, d, h.q_rows, H, d, M, 1, s);
        k_pf_norm_split<<<M, 256, 0, s>>>(H, h.pf_A2, h.pf_rows, w.g2, d, h.eps);
        ok = ok && um_gemm(h, w.wg, h.F, d, h.pf_GU, 2 * h.F, M, 0, s);
        ok = ok && um_gemm(h, w.wu, h.F, d, h.pf_GU + h.F, 2 * h.F, M, 0, s);
        k_pf_silu_split<<<1024, 256, 0, s>>>(P, M);
        ok = ok && um_gemm(h, w.wd, d, h.F, H, d, M, 1, s);
    } else {
        pf_gemm<T>(h.pf_ATT, h.q_rows, w.wo, d, h.q_rows, H, d, M, 1, s);
        k_pf_norm<<<M, 256, 0, s>>>(H, h.pf_XN, w.g2, d, h.eps);
        pf_gemm<T>(h.pf_XN, d, w.wg, h.F, d, h.pf_GU, 2 * h.F, M, 0, s);
        pf_gemm<T>(h.pf_XN, d, w.wu, h.F, d, h.pf_GU + h.F, 2 * h.F, M, 0, s);
        k_pf_silu<<<1024, 256, 0, s>>>(P, M);
        pf_gemm<T>(h.pf_XN, h.F, w.wd, d, h.F, H, d, M, 1, s);
    }
    return ok;
}

template <typename T>
int launch_prefill(const Plan *P, const Plan &h, const int *prompt, int prompt_len, int num_sms, cudaStream_t s) {
    constexpr bool TC = sizeof(T) == 2;
    g_num_sms = num_sms;
    bool ok = true;
    for (int p0 = 0; p0 < prompt_len; p0 += h.pf_rows) {
        const int M = prompt_len - p0 < h.pf_rows ? prompt_len - p0 : h.pf_rows;
        k_pf_embed<T><<<M, 256, 0, s>>>(P, prompt, p0);
        for (int l = 0; l < h.L; ++l) {
            KvT<T> *kc = reinterpret_cast<KvT<T> *>(h.kc) + (long long)l * h.kv_stride;
            KvT<T> *vc = reinterpret_cast<KvT<T> *>(h.vc) + (long long)l * h.kv_stride;
            ok = ok && pf_layer<T>(P, h, h.tl[l], kc, vc, h.pf_H, p0, M, s);
            if (h.aidx[l + 1] >= 0) k_pf_anchor<<<512, 256, 0, s>>>(P, M, h.aidx[l + 1]);
        }
        if (h.Ls > 0) {
            if (TC) {
                const int K = h.nB * h.d;
                k_pf_split<<<1024, 256, 0, s>>>(h.pf_ANCH, K, K, M, h.pf_A2, h.pf_rows);
                ok = ok && um_gemm(h, h.proj, h.d, K, h.pf_Hp, h.d, M, 0, s);
            } else {
                pf_gemm<T>(h.pf_ANCH, h.nB * h.d, h.proj, h.d, h.nB * h.d, h.pf_Hp, h.d, M, 0, s);
            }
            for (int l = 0; l < h.Ls; ++l) {
                KvT<T> *kc = reinterpret_cast<KvT<T> *>(h.pkc) + (long long)l * h.kv_stride;
                KvT<T> *vc = reinterpret_cast<KvT<T> *>(h.pvc) + (long long)l * h.kv_stride;
                ok = ok && pf_layer<T>(P, h, h.pl[l], kc, vc, h.pf_Hp, p0, M, s);
            }
        }
        if (p0 + M == prompt_len)
            k_pf_logits<T><<<1024, 256, h.d * sizeof(float), s>>>(P, h.pf_H + (long long)(M - 1) * h.d);
        if (!ok) return 1;
    }
    launch_prefill_finalize<T>(P, prompt_len, s);
    return 0;
}

__global__ void k_rope_table(float2 *tab, int max_seq, int half, int hd, double theta) {
    const long long total = (long long)max_seq * half;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long p = i / half, j = i - p * half;
        const double inv = pow(theta, -2.0 * (double)j / (double)hd);
        const double a = (double)p * inv;
        tab[i] = make_float2((float)cos(a), (float)sin(a));
    }
}

void launch_rope_table(const Plan &h, float theta, cudaStream_t s) {
    k_rope_table<<<256, 256, 0, s>>>(h.rope, h.max_seq, h.hd / 2, h.hd, (double)theta);
}

void set_prefill_attributes() {
    cudaFuncSetAttribute(k_pf_attn<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * PF_KT * 128 * 4);
    cudaFuncSetAttribute(k_pf_logits<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    cudaFuncSetAttribute(k_pf_logits<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    cudaFuncSetAttribute(k_pf_fa<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem_bytes<128>());
    cudaFuncSetAttribute(k_pf_fa<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem_bytes<64>());
    cudaFuncSetAttribute(k_umma_gemm<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, UM_SMEM);
    cudaFuncSetAttribute(k_umma_gemm<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, UM_SMEM);
    cudaFuncSetAttribute(k_umma_gemm<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, UM_SMEM);
}

template int launch_prefill<float>(const Plan *, const Plan &, const int *, int, int, cudaStream_t);
template int launch_prefill<__nv_bfloat16>(const Plan *, const Plan &, const int *, int, int, cudaStream_t);

}  // namespace spd
