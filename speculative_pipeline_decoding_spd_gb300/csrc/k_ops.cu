// Standalone decode attention through the C ABI: the same kernel code the pipeline step
// runs per stage (attn.cuh), on caller-given q, K and V.  Lets users (and the parity
// tests) drive one attention problem without building a whole model handle.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "attn.cuh"

using namespace spd;

namespace {
thread_local std::string g_ops_error;

int ops_fail(int code, const std::string &msg) {
    g_ops_error = msg;
    return code;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Bytes of split-K scratch one call needs: Hkv counters (256-byte padded), then the
// [Hq][chunks][hd + 4] partials.
size_t attn_scratch_bytes(int Hq, int Hkv, int hd, int seq_len) {
    const int nch = (seq_len + ATT_CHUNK - 1) / ATT_CHUNK;
    return align256((size_t)Hkv * sizeof(int)) + (size_t)Hq * nch * att_part_pitch(hd) * sizeof(float);
}

int attn_validate(int dtype, int Hq, int Hkv, int hd, int seq_len, const void *q, const void *k, const void *v,
                  const void *out) {
    if (dtype != SPD_F32 && dtype != SPD_BF16 && dtype != SPD_F16)
        return ops_fail(SPD_EINVAL, "dtype must be SPD_F32, SPD_BF16 or SPD_F16");
    if (Hq < 1 || Hkv < 1 || Hq % Hkv) return ops_fail(SPD_EINVAL, "need Hq % Hkv == 0");
    const int G = Hq / Hkv;
    if (G > 8 || (G & (G - 1))) return ops_fail(SPD_EINVAL, "Hq / Hkv must be 1, 2, 4 or 8");
    if (hd != 64 && hd != 128) return ops_fail(SPD_EINVAL, "head dim must be 64 or 128");
    if (seq_len < 1 || seq_len > 16384) return ops_fail(SPD_EINVAL, "seq_len must be in [1, 16384]");
    if (!q || !k || !v || !out) return ops_fail(SPD_EINVAL, "null pointer");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(out)) % 16)
        return ops_fail(SPD_EINVAL, "q, k, v and out must be 16-byte aligned");
    return SPD_OK;
}

template <typename T>
__global__ void __launch_bounds__(ATT_THREADS, att_min_blocks<T>()) k_attn_direct(AttnArgs<T> a) {
    attn_cta<T>(a, blockIdx.x % a.Hkv, blockIdx.x / a.Hkv);
}

template <typename T>
void attn_launch_t(int Hq, int Hkv, int hd, int seq_len, const float *q, const void *k, const void *v, float *out,
                   float *part, int *cnt, int nch, cudaStream_t s) {
    AttnArgs<T> a{q, nullptr, nullptr, nullptr, const_cast<T *>(reinterpret_cast<const T *>(k)),
                  const_cast<T *>(reinterpret_cast<const T *>(v)), seq_len, out, part, cnt, 0, nch, Hq, Hkv, hd,
                  1.0f / sqrtf((float)hd)};
    const int sm = att_smem_bytes<T>(hd, Hq / Hkv);
    cudaFuncSetAttribute(k_attn_direct<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    k_attn_direct<T><<<dim3(nch * Hkv), ATT_THREADS, sm, s>>>(a);
}

// Launch over (chunks x Hkv) CTAs with scratch = [counters | partials]; counters are
// cleared on the stream first.
int attn_launch(int dtype, int Hq, int Hkv, int hd, int seq_len, const float *q, const void *k, const void *v,
                float *out, char *scratch, cudaStream_t s) {
    const int nch = (seq_len + ATT_CHUNK - 1) / ATT_CHUNK;
    int *cnt = reinterpret_cast<int *>(scratch);
    float *part = reinterpret_cast<float *>(scratch + align256((size_t)Hkv * sizeof(int)));
    cudaError_t e = cudaMemsetAsync(cnt, 0, (size_t)Hkv * sizeof(int), s);
    if (e != cudaSuccess) return ops_fail(SPD_ECUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    if (dtype == SPD_BF16) attn_launch_t<__nv_bfloat16>(Hq, Hkv, hd, seq_len, q, k, v, out, part, cnt, nch, s);
    else if (dtype == SPD_F16) attn_launch_t<__half>(Hq, Hkv, hd, seq_len, q, k, v, out, part, cnt, nch, s);
    else attn_launch_t<float>(Hq, Hkv, hd, seq_len, q, k, v, out, part, cnt, nch, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return ops_fail(SPD_ECUDA, std::string("attention launch: ") + cudaGetErrorString(e));
    return SPD_OK;
}
}  // namespace

extern "C" int spd_attention_scratch_bytes(int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len, size_t *bytes) {
    if (!bytes) return ops_fail(SPD_EINVAL, "bytes is NULL");
    if (Hq < 1 || Hkv < 1 || seq_len < 1 || (hd != 64 && hd != 128)) return ops_fail(SPD_EINVAL, "bad shape");
    *bytes = attn_scratch_bytes(Hq, Hkv, hd, seq_len);
    return SPD_OK;
}

extern "C" int spd_attention_decode(int32_t dtype, int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len,
                                    const float *q, const void *k, const void *v, float *out, void *scratch,
                                    size_t scratch_bytes, void *stream) {
    int rc = attn_validate(dtype, Hq, Hkv, hd, seq_len, q, k, v, out);
    if (rc) return rc;
    if (!scratch || reinterpret_cast<uintptr_t>(scratch) % 256) return ops_fail(SPD_EINVAL, "scratch must be 256-byte aligned");
    if (scratch_bytes < attn_scratch_bytes(Hq, Hkv, hd, seq_len))
        return ops_fail(SPD_ENOMEM, "scratch too small: see spd_attention_scratch_bytes");
    return attn_launch(dtype, Hq, Hkv, hd, seq_len, q, k, v, out, reinterpret_cast<char *>(scratch),
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" const char *spd_ops_last_error(void) { return g_ops_error.c_str(); }

// ---------------------------------------------------------------------------------------
// Scratch-free variant.  Some callers cannot hand out device memory: their allocations are
// all owned by another allocator (a framework's caching allocator, a fixed arena) with no
// spare buffer to lend, or they run where cudaMalloc's implicit device synchronisation is
// not acceptable.  For them the split-K scratch lives in this file-scope array, reserved
// on every GPU that loads the library until the process exits.  Calls share it: each call
// clears the arrival counters it needs, the partials need no clearing, and two calls
// that run at the same time on the GPU race on it.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(1) << 20;   // 1 MiB
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the array on the current device, looked up once per device.  In host
// code the array's name is only a stand-in; the kernel must get this address.
int noalloc_scratch(char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ops_fail(SPD_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return ops_fail(SPD_EINVAL, "device index above 63");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return ops_fail(SPD_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = reinterpret_cast<char *>(g_noalloc_ptr[dev]);
    return SPD_OK;
}
}  // namespace

extern "C" int spd_attention_decode_noalloc(int32_t dtype, int32_t Hq, int32_t Hkv, int32_t hd, int32_t seq_len,
                                            const float *q, const void *k, const void *v, float *out, void *stream) {
    int rc = attn_validate(dtype, Hq, Hkv, hd, seq_len, q, k, v, out);
    if (rc) return rc;
    const size_t need = attn_scratch_bytes(Hq, Hkv, hd, seq_len);
    if (need > NOALLOC_SCRATCH_BYTES)
        return ops_fail(SPD_ECAPACITY, "spd_attention_decode_noalloc: this shape needs " + std::to_string(need) +
                                           " bytes of scratch, the built-in buffer holds " +
                                           std::to_string(NOALLOC_SCRATCH_BYTES) +
                                           "; use spd_attention_decode with caller scratch");
    char *scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return attn_launch(dtype, Hq, Hkv, hd, seq_len, q, k, v, out, scratch, reinterpret_cast<cudaStream_t>(stream));
}
