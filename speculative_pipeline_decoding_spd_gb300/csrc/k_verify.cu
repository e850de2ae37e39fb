// Streaming verification, commit, rollback and reseed of one pipeline step (one CTA,
// on the device: no host round trip per step).
//
// Speculative pipeline decoding, machine review "What carries the argument":
// verification is streaming — the token leaving the last stage yields the target's
// prediction for the next position, which checks the draft one stage behind it; on a
// rejection the KV cache is truncated after the exiting token, the pipeline is flushed
// and stage 0 is reseeded with the target's token.  At T > 0 the check is speculative
// rejection sampling (review "Assumptions", section 3.5, after Leviathan et al.): keep
// the draft x with probability min(1, p_T(x) / p_D(x)), else draw from the normalised
// residual max(0, p_T - p_D).
//
// Philox stream (the pages only say the uniforms come from a seeded Philox): counter (t, purpose),
// purposes 0 draft sample, 1 keep test, 2 target / residual sample, 3 forced coin,
// 4 forced alternative id; u = (word >> 8) * 2^-24.
#include "common.cuh"

namespace spd {

constexpr int VT = 512;   // verify kernel threads

__device__ __forceinline__ float u01(uint32_t w) { return (float)(w >> 8) * (1.0f / 16777216.0f); }

// Block-wide inverse-CDF draw over weights w(i), i in [0, V): the smallest i whose running
// sum (index order) exceeds u * total.  The ids are cut into tiles of 512 (16 per lane of a
// warp): pass 1, each warp sums its tiles (tiles w, w + nw, ...; lane l reads ids l, l + 32,
// ..., coalesced) with no block-wide barrier inside the loop; warp 0 then runs the running
// sum over the tile totals in tile order (32 tiles per warp-wide scan), and scans the
// crossing tile again with lane l owning the contiguous slice [16 l, 16 l + 16).
// The weight functor has two parts, ld(i) (the global loads id i needs, as a float2) and
// w(f) (the arithmetic): a lane issues all 16 loads of a tile before it computes any weight,
// so a tile costs one memory latency, not sixteen.
// Returns the index in all threads; *total_out receives the total.
constexpr int SAMPLE_PER = 16;
constexpr int SAMPLE_TILE = 32 * SAMPLE_PER;
constexpr int SAMPLE_MAX_TILES = 512;   // V up to 262144

__device__ __forceinline__ float warp_incl_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// weight exp(z_i / T - m) of a softmax draw (m the row's max of z / T)
struct SoftmaxW {
    const float *z;
    float invT, m;
    __device__ __forceinline__ float2 ld(int i) const { return make_float2(z[i], 0.f); }
    __device__ __forceinline__ float w(float2 f) const { return expf(f.x * invT - m); }
};
// weight max(0, p_T(i) - p_D(i)) of the residual draw; rt, rd the reciprocals of the two
// rows' sums of exp(z / T - max)
struct ResidualW {
    const float *zt, *zd;
    float invT, mt, rt, md, rd;
    __device__ __forceinline__ float2 ld(int i) const { return make_float2(zt[i], zd[i]); }
    __device__ __forceinline__ float w(float2 f) const {
        return fmaxf(expf(f.x * invT - mt) * rt - expf(f.y * invT - md) * rd, 0.f);
    }
};

template <typename WF>
__device__ int block_sample(int V, float u, const WF &wf, float *red, float *total_out) {
    __shared__ float s_tile[SAMPLE_MAX_TILES];
    __shared__ int s_pick;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int ntiles = (V + SAMPLE_TILE - 1) / SAMPLE_TILE;
    for (int t = warp; t < ntiles; t += nw) {
        const int base = t * SAMPLE_TILE;
        float2 f[SAMPLE_PER];
#pragma unroll
        for (int j = 0; j < SAMPLE_PER; ++j) {
            const int i = base + j * 32 + lane;
            f[j] = i < V ? wf.ld(i) : make_float2(0.f, 0.f);
        }
        float loc = 0.f;
#pragma unroll
        for (int j = 0; j < SAMPLE_PER; ++j)
            if (base + j * 32 + lane < V) loc += wf.w(f[j]);
        loc = warp_sum(loc);
        if (lane == 0) s_tile[t] = loc;
    }
    __syncthreads();
    if (warp == 0) {
        float tot = 0.f;
        for (int t = lane; t < ntiles; t += 32) tot += s_tile[t];
        tot = warp_sum(tot);
        const float target = u * tot;
        // the crossing tile
        float before = 0.f;
        int ct = -1;
        for (int t0 = 0; t0 < ntiles; t0 += 32) {
            const int t = t0 + lane;
            const float w = t < ntiles ? s_tile[t] : 0.f;
            const float inc = warp_incl_scan(w);
            const unsigned hit = __ballot_sync(0xffffffffu, t < ntiles && w > 0.f && before + inc > target);
            if (hit) {
                const int l = __ffs(hit) - 1;
                before += __shfl_sync(0xffffffffu, inc - w, l);
                ct = t0 + l;
                break;
            }
            before += __shfl_sync(0xffffffffu, inc, 31);
        }
        int pick = -1, lastnz = -1;
        if (ct < 0) {
            // rounding left the target beyond the running sum: the last id with weight
            ct = ntiles - 1;
            for (int t = ntiles - 1; t >= 0; --t)
                if (s_tile[t] > 0.f) { ct = t; break; }
            before = -INFINITY;   // every weighted id below crosses; the scan below keeps the last
        }
        // the crossing tile, lane l owning ids [16 l, 16 l + 16) of it
        const int lo = ct * SAMPLE_TILE + lane * SAMPLE_PER;
        float2 f[SAMPLE_PER];
        float w[SAMPLE_PER], sl = 0.f;
#pragma unroll
        for (int j = 0; j < SAMPLE_PER; ++j) f[j] = lo + j < V ? wf.ld(lo + j) : make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < SAMPLE_PER; ++j) {
            w[j] = lo + j < V ? wf.w(f[j]) : 0.f;
            sl += w[j];
        }
        const float inc = warp_incl_scan(sl);
        const unsigned hit = __ballot_sync(0xffffffffu, sl > 0.f && before + inc > target);
        const unsigned nz = __ballot_sync(0xffffffffu, sl > 0.f);
        const int hl = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : 0);
        if (lane == hl) {
            float acc = before == -INFINITY ? 0.f : before + inc - sl;
            for (int j = 0; j < SAMPLE_PER; ++j) {
                if (w[j] > 0.f) lastnz = lo + j;
                acc += w[j];
                if (hit && acc > target && w[j] > 0.f) {
                    pick = lo + j;
                    break;
                }
            }
            s_pick = pick >= 0 ? pick : (lastnz >= 0 ? lastnz : min(lo, V - 1));
            red[0] = tot;
        }
    }
    __syncthreads();
    if (total_out) *total_out = red[0];
    const int pick = s_pick;
    __syncthreads();
    return pick;
}

// max and sum of exp(z/T - max) over a logits row in one coalesced pass: each thread keeps a
// running max and a sum rescaled when its max grows, then the threads' pairs are merged by a
// fixed tree
__device__ void softmax_stats(const float *z, int V, float invT, float *red, float *m_out, float *s_out) {
    float m = -INFINITY, sum = 0.f;
    for (int i0 = threadIdx.x; i0 < V; i0 += 4 * blockDim.x) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * blockDim.x;
            v[j] = i < V ? z[i] * invT : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (v[j] > m) {
                sum = sum * expf(m - v[j]);
                m = v[j];
            }
            if (v[j] > -INFINITY) sum += expf(v[j] - m);
        }
    }
    const float M = block_max(m, red);
    const float S = block_sum(m == -INFINITY ? 0.f : sum * expf(m - M), red);
    *m_out = M;
    *s_out = S;
}

template <typename T>
__device__ void embed_into_slot(const Plan *__restrict__ P, int slot, int tok) {
    const int d = P->d;
    const T *e = reinterpret_cast<const T *>(P->embed) + (long long)tok * d;
    float *x = P->X + (long long)slot * d;
    float *a0 = P->ANCH + (long long)slot * P->nB * d;
    __nv_bfloat16 *b0 = P->ANCHb + (long long)slot * P->nB * d;
    const long long blo = (long long)(P->n + 1) * P->nB * d;   // lo parts (zero: an embedding row is bf16)
    // 8 elements per thread and pass: one 16-byte load of a bf16 row (two of an fp32 row), all
    // of a thread's loads issued before its stores (d is a multiple of 64)
    for (int k0 = 8 * threadIdx.x; k0 < d; k0 += 8 * blockDim.x) {
        float v[8];
        if constexpr (sizeof(T) == 2) {
            const uint4 w = *reinterpret_cast<const uint4 *>(e + k0);
            v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
            v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
            *reinterpret_cast<uint4 *>(b0 + k0) = w;                               // the hi parts are the row itself
            *reinterpret_cast<uint4 *>(b0 + blo + k0) = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const float4 f0 = *reinterpret_cast<const float4 *>(e + k0);
            const float4 f1 = *reinterpret_cast<const float4 *>(e + k0 + 4);
            v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w; v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
        }
        const float4 o0 = make_float4(v[0], v[1], v[2], v[3]), o1 = make_float4(v[4], v[5], v[6], v[7]);
        *reinterpret_cast<float4 *>(x + k0) = o0;
        *reinterpret_cast<float4 *>(x + k0 + 4) = o1;
        *reinterpret_cast<float4 *>(a0 + k0) = o0;
        *reinterpret_cast<float4 *>(a0 + k0 + 4) = o1;
    }
}

template <typename T>
__global__ void __launch_bounds__(VT) k_verify(const Plan *__restrict__ P) {
    __shared__ float red[40];
    __shared__ int s_done, s_t, s_head, s_ex, s_q, s_x, s_xslot, s_P0, s_newslot, s_draft, s_y, s_ok, s_active;
    __shared__ float s_tmax, s_tsum;
    // The slot state is small (about 1.2 KB): every thread loads a piece of it into shared
    // memory at once, thread 0's decisions below work on that copy (no chain of dependent
    // global loads), and all threads write it back before the next step's embedding.
    __shared__ __align__(16) DevState sst;
    __shared__ int s_err0;
    static_assert(sizeof(DevState) % 16 == 0, "state copied in 16-byte words");
    DevState *const gst = P->st;
    pdl_wait();   // logits and argmax of the LM head launch
    pdl_trigger();
    for (int i = threadIdx.x; i < (int)(sizeof(DevState) / 16); i += blockDim.x)
        reinterpret_cast<uint4 *>(&sst)[i] = reinterpret_cast<const uint4 *>(gst)[i];
    __syncthreads();
    const int n = P->n, ns = n + 1, V = P->V;
    const float T_ = P->temperature;
    DevState *st = &sst;
    if (threadIdx.x == 0) {
        s_err0 = st->error;
        s_done = st->done;
        if (!s_done) {
            const int t = st->t + 1;
            st->t = t;
            const int head = st->head;
            s_t = t;
            s_head = head;
            const int s0 = ring(head, 0, ns);
            s_P0 = st->pos[s0];
            s_newslot = ring(head + 1, 0, ns);
            const int exs = ring(head, n - 1, ns);
            s_ex = st->valid[exs];
            s_q = st->pos[exs];
            if (n >= 2) {
                s_xslot = ring(head, n - 2, ns);
                s_x = st->tok[s_xslot];
            } else {
                s_xslot = s_newslot;
                s_x = -1;   // the new draft (set below)
            }
            // KV valid lengths of the layers that ran, and the bytes streamed
            int active = 0;
            for (int s = 0; s < n; ++s) {
                const int slot = ring(head, s, ns);
                if (!st->valid[slot]) continue;
                ++active;
                for (int l = P->b[s]; l < P->b[s + 1]; ++l) st->len[l] = st->pos[slot] + 1;
                st->weight_bytes += (double)P->layer_bytes * (P->b[s + 1] - P->b[s]);
            }
            st->weight_bytes += (double)(P->pdm_bytes + P->lm_bytes);
            s_active = active;
        }
    }
    __syncthreads();
    if (s_done) return;
    const int t = s_t;
    // ---- the draft for position P0+1
    if (threadIdx.x == 0) {
        int draft;
        if (P->forced) {
            const int idx = s_P0 + 1;
            int r = 0;
            if (idx < P->forced_ref_len) r = P->forced_ref[idx];
            else st->error = ERR_FORCED_REF;
            const uint32_t c = philox_word0((uint32_t)t, 3u, P->seed_lo, P->seed_hi) >> 8;
            if (c < P->forced_thr) {
                draft = r;
            } else {
                const uint32_t a = philox_word0((uint32_t)t, 4u, P->seed_lo, P->seed_hi) >> 8;
                const unsigned long long alt = ((unsigned long long)a * (unsigned long long)(V - 1)) >> 24;
                draft = (int)(((long long)r + 1 + (long long)alt) % V);
            }
        } else {
            draft = st->top[1];
        }
        s_draft = draft;
    }
    __syncthreads();
    if (!P->forced && T_ > 0.f) {
        // sample the draft from softmax(z_D / T) and keep its normalisers with the slot (the
        // tensor-core LM head has drawn it already, from the same uniform)
        if (P->lm_stats) {
            if (threadIdx.x == 0) {
                s_draft = st->samp;
                st->dmax[s_newslot] = st->lmM[1];
                st->dsum[s_newslot] = st->lmS[1];
            }
        } else {
            const float *zd = P->dlogits + (long long)s_newslot * V;
            const float invT = 1.0f / T_;
            float m, s;
            softmax_stats(zd, V, invT, red, &m, &s);
            const float u0 = u01(philox_word0((uint32_t)t, 0u, P->seed_lo, P->seed_hi));
            const int pick = block_sample(V, u0, SoftmaxW{zd, invT, m}, red + 4, nullptr);
            if (threadIdx.x == 0) {
                s_draft = pick;
                st->dmax[s_newslot] = m;
                st->dsum[s_newslot] = s;
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0 && n == 1) s_x = s_draft;
    __syncthreads();
    // ---- verify the draft behind the exiting token
    if (s_ex) {
        if (T_ == 0.f) {
            if (threadIdx.x == 0) {
                s_y = st->top[0];
                s_ok = (s_x == s_y);
            }
            __syncthreads();
        } else {
            const float invT = 1.0f / T_;
            const float *zt = P->logits;
            const float *zd = P->dlogits + (long long)s_xslot * V;
            float tm, ts;
            if (P->lm_stats) {
                tm = st->lmM[0];
                ts = st->lmS[0];
            } else {
                softmax_stats(zt, V, invT, red, &tm, &ts);
            }
            if (threadIdx.x == 0) {
                const int x = s_x;
                const float pt = expf(zt[x] * invT - tm) / ts;
                const float pd = expf(zd[x] * invT - st->dmax[s_xslot]) / st->dsum[s_xslot];
                const float u1 = u01(philox_word0((uint32_t)t, 1u, P->seed_lo, P->seed_hi));
                s_ok = (u1 < pt / pd);
                s_tmax = tm;
                s_tsum = ts;
            }
            __syncthreads();
            if (!s_ok) {
                const float dm = st->dmax[s_xslot], ds = st->dsum[s_xslot];
                const float tmx = s_tmax, tsm = s_tsum;
                const float u2 = u01(philox_word0((uint32_t)t, 2u, P->seed_lo, P->seed_hi));
                float tot;
                int y = block_sample(V, u2, ResidualW{zt, zd, invT, tmx, 1.0f / tsm, dm, 1.0f / ds}, red + 4, &tot);
                if (!(tot > 0.f)) y = block_sample(V, u2, SoftmaxW{zt, invT, tmx}, red + 4, nullptr);
                if (threadIdx.x == 0) s_y = y;
            } else if (threadIdx.x == 0) {
                s_y = s_x;
            }
            __syncthreads();
        }
    }
    // ---- commit / rollback / reseed / shift / trace
    if (threadIdx.x == 0) {
        const int head = s_head, nh = head + 1;
        const int ytarget = s_ex ? s_y : -1;
        int commit = -1, accept = -1;
        bool flushed = false;
        if (s_ex) {
            accept = s_ok;
            commit = s_ok ? s_x : s_y;
            st->N += 1;
            if (st->N < P->max_new) P->out_tokens[st->N] = commit;
            st->pending = 1;
            st->pdm_len = s_q + 1;
            if (s_ok) {
                st->accepts += 1;
                st->run_cur += 1;
            } else {
                st->rejects += 1;
                st->run_sum += st->run_cur;
                st->run_count += 1;
                st->run_cur = 0;
                flushed = true;
                for (int l = 0; l < P->L; ++l) st->len[l] = s_q + 1;
            }
        } else {
            st->pending = 0;
        }
        const int ns0 = ring(nh, 0, ns);
        int newpos, newtok;
        if (flushed) {
            newpos = s_q + 1;
            newtok = s_y;
            for (int s = 1; s < n; ++s) st->valid[ring(nh, s, ns)] = 0;
        } else {
            newpos = s_P0 + 1;
            newtok = s_draft;
        }
        if (newpos >= P->max_seq) {
            st->error = ERR_SEQ_FULL;
            st->done = 1;
            newpos = P->max_seq - 1;
        }
        if (newtok < 0 || newtok >= V) {
            st->error = ERR_TOKEN;
            newtok = 0;
        }
        st->valid[ns0] = 1;
        st->pos[ns0] = newpos;
        st->tok[ns0] = newtok;
        st->head = nh;
        s_newslot = ns0;
        s_y = newtok;
        if (t - 1 < P->max_steps) {
            spd_trace_rec rec;
            rec.t = t;
            rec.exit_pos = s_ex ? s_q : -1;
            rec.draft = s_ex ? s_x : -1;
            rec.target = ytarget;
            rec.accept = accept;
            rec.commit = commit;
            rec.pdm_top = st->top[1];
            rec.new_draft = s_draft;
            rec.n_committed = st->N;
            rec.n_active = s_active;
            rec.target_logit = st->topval[0];
            rec.pdm_logit = st->topval[1];
            P->trace[t - 1] = rec;
            for (int l = 0; l < P->L; ++l) P->trace_len[(long long)(t - 1) * P->L + l] = st->len[l];
        } else {
            st->error = ERR_TRACE_FULL;
            st->done = 1;
        }
        if (1 + st->N >= P->max_new) st->done = 1;
    }
    __syncthreads();
    // write the state back: all 16-byte words but the first two (which hold the error
    // word, written only if this kernel changed it), then the first eight ints
    for (int i = 2 + threadIdx.x; i < (int)(sizeof(DevState) / 16); i += blockDim.x)
        reinterpret_cast<uint4 *>(P->st)[i] = reinterpret_cast<const uint4 *>(&sst)[i];
    if (threadIdx.x < 8) {
        const int *src = reinterpret_cast<const int *>(&sst);
        int *dst = reinterpret_cast<int *>(P->st);
        if (threadIdx.x != 5 || sst.error != s_err0) dst[threadIdx.x] = src[threadIdx.x];
    }
    embed_into_slot<T>(P, s_newslot, s_y);
}

// First token after the prefill (greedy argmax, or a draw with uniform (0, purpose 2)),
// then the initial pipeline state: y0 committed and seeded into stage 0 (slot 0).
template <typename T>
__global__ void __launch_bounds__(VT) k_prefill_finalize(const Plan *__restrict__ P, int prompt_len) {
    __shared__ float red[40];
    __shared__ float s_bv[VT / 32];
    __shared__ int s_bi[VT / 32];
    __shared__ int s_y;
    DevState *st = P->st;
    const int V = P->V;
    const float *z = P->pf_logits;
    if (P->temperature > 0.f) {
        const float invT = 1.0f / P->temperature;
        float m, s;
        softmax_stats(z, V, invT, red, &m, &s);
        const float u = u01(philox_word0(0u, 2u, P->seed_lo, P->seed_hi));
        const int y = block_sample(V, u, SoftmaxW{z, invT, m}, red + 4, nullptr);
        if (threadIdx.x == 0) s_y = y;
    } else {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = threadIdx.x; i < V; i += blockDim.x) {
            const float v = z[i];
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((threadIdx.x & 31) == 0) { s_bv[threadIdx.x >> 5] = bv; s_bi[threadIdx.x >> 5] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            float b = -INFINITY;
            int id = 0x7fffffff;
            for (int w = 0; w < VT / 32; ++w)
                if (s_bv[w] > b || (s_bv[w] == b && s_bi[w] < id)) { b = s_bv[w]; id = s_bi[w]; }
            s_y = id;
            st->topval[0] = b;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int y0 = s_y;
        st->head = 0;
        st->t = 0;
        st->N = 0;
        st->done = P->max_new <= 1 ? 1 : 0;
        st->pending = 0;
        st->error = 0;
        st->pdm_len = prompt_len;
        st->prompt_len = prompt_len;
        for (int i = 0; i < MAXS; ++i) st->valid[i] = 0;
        st->valid[0] = 1;
        st->pos[0] = prompt_len;
        st->tok[0] = y0;
        for (int l = 0; l < P->L; ++l) st->len[l] = prompt_len;
        st->top[0] = y0;
        st->top[1] = -1;
        st->accepts = st->rejects = st->run_cur = st->run_sum = st->run_count = 0;
        st->weight_bytes = 0.0;
        P->out_tokens[0] = y0;
    }
    __syncthreads();
    embed_into_slot<T>(P, 0, s_y);
}

template <typename T>
void launch_verify(const Plan *P, const Plan &h, cudaStream_t s) {
    launch_k(k_verify<T>, dim3(1), dim3(VT), 0, s, h.pdl != 0, P);
}
template <typename T>
void launch_prefill_finalize(const Plan *P, int prompt_len, cudaStream_t s) {
    k_prefill_finalize<T><<<1, VT, 0, s>>>(P, prompt_len);
}
template void launch_verify<float>(const Plan *, const Plan &, cudaStream_t);
template void launch_verify<__nv_bfloat16>(const Plan *, const Plan &, cudaStream_t);
template void launch_prefill_finalize<float>(const Plan *, int, cudaStream_t);
template void launch_prefill_finalize<__nv_bfloat16>(const Plan *, int, cudaStream_t);

}  // namespace spd
