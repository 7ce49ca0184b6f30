// kda_api.cu -- the extern "C" entry points of libkda (declared in include/kda.h).
//
// Host-side argument checks, the per-device error word, and the launches.  No
// CUDA allocation happens here; every buffer is the caller's.
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

// One error word per device: kernels record the first error they meet, the
// host reads and clears it in kda_get_last_device_error().
__device__ unsigned int g_device_error_word;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    unsigned int *error_word = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

// Looks up (once per device) the SM count, whether the device is an sm_103
// part this library was built for, and the device address of the error word.
kda_status current_device(DeviceInfo **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    DeviceInfo &info = g_devices[dev];
    if (!info.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_NO_DEVICE;
        }
        info.supported = (prop.major == 10 && prop.minor == 3);
        info.num_sms = prop.multiProcessorCount;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error_word) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        info.error_word = static_cast<unsigned int *>(addr);
        info.ready = true;
    }
    if (!info.supported) return KDA_ERR_NO_DEVICE;
    *out = &info;
    return KDA_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_dtype(kda_dtype d) { return d == KDA_BF16 || d == KDA_FP32; }

// Whether two byte ranges share an address.
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return a != nullptr && b != nullptr && na > 0 && nb > 0 && pa < pb + nb && pb < pa + na;
}

kda_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    cudaGetLastError();
    return KDA_ERR_CUDA;
}

// Host checks of kda_chunk_prefill's arguments other than the workspace.
kda_status check_prefill_args(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const int32_t *cu_seqlens, int B, int64_t N,
                              int H, int K, int V, const float *initial_state,
                              const float *final_state, const void *o, kda_dtype o_dtype) {
    if (N < 0 || B < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(o_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (cu_seqlens == nullptr && B != 1) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(o) || !aligned16(initial_state) || !aligned16(final_state) ||
        !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    return KDA_OK;
}

}  // namespace

namespace kda {

cudaError_t ensure_dynamic_smem(const void *func, int bytes) {
    struct Done {
        int dev;
        const void *func;
        int bytes;
    };
    static std::mutex m;
    static std::vector<Done> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(m);
    for (const Done &d : done)
        if (d.dev == dev && d.func == func && d.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back(Done{dev, func, bytes});
    return e;
}

}  // namespace kda

extern "C" {

int kda_version(void) { return KDA_VERSION; }

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED_SHAPE: return "KDA_ERR_UNSUPPORTED_SHAPE";
        case KDA_ERR_UNSUPPORTED_DTYPE: return "KDA_ERR_UNSUPPORTED_DTYPE";
        case KDA_ERR_MISALIGNED: return "KDA_ERR_MISALIGNED";
        case KDA_ERR_WORKSPACE_TOO_SMALL: return "KDA_ERR_WORKSPACE_TOO_SMALL";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT";
        case KDA_ERR_NONFINITE: return "KDA_ERR_NONFINITE";
        case KDA_ERR_NOT_IMPLEMENTED: return "KDA_ERR_NOT_IMPLEMENTED";
        case KDA_ERR_NO_DEVICE: return "KDA_ERR_NO_DEVICE";
        case KDA_ERR_DECAY_RANGE: return "KDA_ERR_DECAY_RANGE";
    }
    return "KDA_ERR_UNKNOWN";
}

kda_status kda_gate_fused(const void *f, kda_dtype f_dtype, const void *b, kda_dtype b_dtype,
                          const float *A_log, kda_alog_mode alog_mode, const float *dt_bias,
                          float *g_out, float *beta_out, int64_t N, int H, int K, void *stream) {
    if (N < 0 || H < 1 || K < 1) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(f_dtype) || !valid_dtype(b_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (alog_mode != KDA_ALOG_PER_HEAD && alog_mode != KDA_ALOG_PER_CHANNEL &&
        alog_mode != KDA_ALOG_PER_HEAD_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if ((b == nullptr) != (beta_out == nullptr)) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || g_out == nullptr)) return KDA_ERR_INVALID_ARG;
    if (A_log == nullptr || dt_bias == nullptr) return KDA_ERR_INVALID_ARG;
    if (!aligned16(f) || !aligned16(b) || !aligned16(A_log) || !aligned16(dt_bias) ||
        !aligned16(g_out) || !aligned16(beta_out))
        return KDA_ERR_MISALIGNED;
    if (N == 0) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_gate(f, f_dtype == KDA_BF16, b, b_dtype == KDA_BF16, A_log,
                                      static_cast<int>(alog_mode), dt_bias, g_out, beta_out, N, H,
                                      K, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_prefill_workspace_size(int64_t N, int B, int H, int K, int V) {
    if (N < 0 || B < 1 || H < 1 || K != 128 || V != 128) return 0;
    return kda::prefill_workspace_bytes(N, B, H);
}

kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const int32_t *cu_seqlens, int B, int64_t N, int H,
                             int K, int V, float scale, const float *initial_state,
                             float *final_state, void *o, kda_dtype o_dtype, void *workspace,
                             size_t workspace_bytes, void *stream) {
    kda_status st = check_prefill_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, initial_state,
                                       final_state, o, o_dtype);
    if (st != KDA_OK) return st;
    if (!aligned16(workspace)) return KDA_ERR_MISALIGNED;
    const size_t need = kda::prefill_workspace_bytes(N, B, H);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_prefill(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, B, N, H, scale, initial_state,
        final_state, o, o_dtype == KDA_BF16, workspace, dev->error_word, dev->num_sms,
        static_cast<cudaStream_t>(stream)));
}

kda_status kda_chunk_prefill_gated(const void *q, const void *k, const void *v, const void *f,
                                   kda_dtype f_dtype, const void *b, kda_dtype b_dtype,
                                   const float *A_log, kda_alog_mode alog_mode,
                                   const float *dt_bias, const int32_t *cu_seqlens, int B,
                                   int64_t N, int H, int K, int V, float scale,
                                   const float *initial_state, float *final_state, void *o,
                                   kda_dtype o_dtype, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (N < 0 || B < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(o_dtype) || !valid_dtype(b_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (f_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (alog_mode != KDA_ALOG_PER_HEAD && alog_mode != KDA_ALOG_PER_CHANNEL &&
        alog_mode != KDA_ALOG_PER_HEAD_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && B != 1) return KDA_ERR_INVALID_ARG;
    if (A_log == nullptr || dt_bias == nullptr) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (q == nullptr || k == nullptr || v == nullptr || f == nullptr || b == nullptr ||
                  o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(f) || !aligned16(b) ||
        !aligned16(A_log) || !aligned16(dt_bias) || !aligned16(o) || !aligned16(initial_state) ||
        !aligned16(final_state) || !aligned16(workspace) || !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    const size_t need = kda::prefill_workspace_bytes(N, B, H);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_prefill_gated(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), static_cast<const __nv_bfloat16 *>(f), b,
        b_dtype == KDA_BF16, A_log, static_cast<int>(alog_mode), dt_bias, cu_seqlens, B, N, H,
        scale, initial_state, final_state, o, o_dtype == KDA_BF16, workspace, dev->error_word,
        dev->num_sms, static_cast<cudaStream_t>(stream)));
}

kda_status kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const int32_t *cu_seqlens, int B,
                                     int64_t N, int H, int K, int V, float scale,
                                     const float *initial_state, float *final_state, void *o,
                                     kda_dtype o_dtype, void *stream) {
    // The same argument and device checks as kda_chunk_prefill, in the same
    // order, before the scratch lookup, so both return the same status codes.
    kda_status st = check_prefill_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, initial_state,
                                       final_state, o, o_dtype);
    if (st != KDA_OK) return st;
    DeviceInfo *dev = nullptr;
    st = current_device(&dev);
    if (st != KDA_OK) return st;
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    if (kda::builtin_prefill_scratch(&scratch, &scratch_bytes) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    if (kda::prefill_workspace_bytes(N, B, H) > scratch_bytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
    return kda_chunk_prefill(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, scale, initial_state,
                             final_state, o, o_dtype, scratch, scratch_bytes, stream);
}

kda_status kda_recurrent_decode(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float *state, int B, int H, int K, int V,
                                float scale, void *o, kda_dtype o_dtype, void *stream) {
    if (B < 0 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(o_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (B > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || state == nullptr || o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(state) || !aligned16(o))
        return KDA_ERR_MISALIGNED;
    if (B == 0) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_decode(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, state, B, H, scale, o,
        o_dtype == KDA_BF16, static_cast<cudaStream_t>(stream)));
}

kda_status kda_recurrent_decode_indexed(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta, void *state_pool,
                                        kda_dtype state_dtype, const int32_t *state_indices,
                                        int num_slots, int B, int H, int K, int V, float scale,
                                        void *o, kda_dtype o_dtype, void *stream) {
    if (B < 0 || H < 1 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(o_dtype) || !valid_dtype(state_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (B > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || state_pool == nullptr || state_indices == nullptr ||
                  o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(state_pool) || !aligned16(state_indices) || !aligned16(o))
        return KDA_ERR_MISALIGNED;
    if (B == 0) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_decode_indexed(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, state_pool, state_dtype == KDA_BF16,
        state_indices, num_slots, B, H, scale, o, o_dtype == KDA_BF16, dev->error_word,
        static_cast<cudaStream_t>(stream)));
}

kda_status kda_recurrent_decode_gated(const void *q, const void *k, const void *v,
                                      const void *f, kda_dtype f_dtype, const void *b,
                                      kda_dtype b_dtype, const float *A_log,
                                      kda_alog_mode alog_mode, const float *dt_bias,
                                      void *state_pool, kda_dtype state_dtype,
                                      const int32_t *state_indices, int num_slots, int B, int H,
                                      int K, int V, float scale, void *o, kda_dtype o_dtype,
                                      void *stream) {
    if (B < 0 || H < 1 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (state_indices == nullptr && num_slots < B) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(o_dtype) || !valid_dtype(state_dtype) || !valid_dtype(f_dtype) ||
        !valid_dtype(b_dtype))
        return KDA_ERR_UNSUPPORTED_DTYPE;
    if (alog_mode != KDA_ALOG_PER_HEAD && alog_mode != KDA_ALOG_PER_CHANNEL &&
        alog_mode != KDA_ALOG_PER_HEAD_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if (B > 0 && (q == nullptr || k == nullptr || v == nullptr || f == nullptr || b == nullptr ||
                  A_log == nullptr || dt_bias == nullptr || state_pool == nullptr ||
                  o == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(f) || !aligned16(b) ||
        !aligned16(state_pool) || !aligned16(state_indices) || !aligned16(o))
        return KDA_ERR_MISALIGNED;
    if (B == 0) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_decode_gated(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), f, f_dtype == KDA_BF16, b, b_dtype == KDA_BF16,
        A_log, static_cast<int>(alog_mode), dt_bias, state_pool, state_dtype == KDA_BF16,
        state_indices, state_indices == nullptr ? B : num_slots, B, H, scale, o,
        o_dtype == KDA_BF16, dev->error_word, static_cast<cudaStream_t>(stream)));
}

size_t kda_gate_backward_workspace_size(int64_t N, int H, int K) {
    return kda::gate_bwd_workspace_bytes(N, H, K);
}

kda_status kda_gate_backward(const void *f, kda_dtype f_dtype, const void *b, kda_dtype b_dtype,
                             const float *A_log, kda_alog_mode alog_mode, const float *dt_bias,
                             const float *dg, const float *dbeta, float *df, float *db,
                             float *dA_log, float *ddt_bias, int64_t N, int H, int K,
                             void *workspace, size_t workspace_bytes, void *stream) {
    if (N < 0 || H < 1 || K < 1) return KDA_ERR_INVALID_ARG;
    if (K % 8 != 0) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(f_dtype) || !valid_dtype(b_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (alog_mode != KDA_ALOG_PER_HEAD && alog_mode != KDA_ALOG_PER_CHANNEL &&
        alog_mode != KDA_ALOG_PER_HEAD_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    const bool with_beta = b != nullptr;
    if (with_beta != (dbeta != nullptr) || with_beta != (db != nullptr)) return KDA_ERR_INVALID_ARG;
    if (A_log == nullptr || dt_bias == nullptr) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (f == nullptr || dg == nullptr || df == nullptr)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(f) || !aligned16(dg) || !aligned16(df) || !aligned16(workspace))
        return KDA_ERR_MISALIGNED;
    if (workspace == nullptr || workspace_bytes < kda::gate_bwd_workspace_bytes(N, H, K))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    return from_cuda(kda::launch_gate_backward(
        f, f_dtype == KDA_BF16, b, b_dtype == KDA_BF16, A_log, static_cast<int>(alog_mode),
        dt_bias, dg, dbeta, df, db, dA_log, ddt_bias, N, H, K, workspace,
        static_cast<cudaStream_t>(stream)));
}

kda_status kda_short_conv_qkv(const void *x_q, const void *x_k, const void *x_v,
                              const float *w_q, const float *w_k, const float *w_v,
                              const int32_t *cu_seqlens, int B, int64_t N, int C,
                              const void *conv_state_in, void *conv_state_out,
                              void *q, void *k, void *v, void *stream) {
    if (N < 0 || B < 1 || (cu_seqlens == nullptr && B != 1)) return KDA_ERR_INVALID_ARG;
    if (C < 128 || C % 128 != 0) return KDA_ERR_UNSUPPORTED_SHAPE;
    const void *xs[3] = {x_q, x_k, x_v};
    const float *ws[3] = {w_q, w_k, w_v};
    void *ys[3] = {q, k, v};
    const size_t tok_bytes = static_cast<size_t>(N) * C * 2;
    const size_t st_bytes = static_cast<size_t>(B) * 9 * C * 2;
    if (N > 0) {
        for (int i = 0; i < 3; ++i)
            if (xs[i] == nullptr || ws[i] == nullptr || ys[i] == nullptr) return KDA_ERR_INVALID_ARG;
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j) {
                if (overlaps(ys[i], tok_bytes, xs[j], tok_bytes)) return KDA_ERR_INVALID_ARG;
                if (i < j && overlaps(ys[i], tok_bytes, ys[j], tok_bytes)) return KDA_ERR_INVALID_ARG;
            }
    }
    if (overlaps(conv_state_in, st_bytes, conv_state_out, st_bytes)) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (!aligned16(xs[i]) || !aligned16(ws[i]) || !aligned16(ys[i])) return KDA_ERR_MISALIGNED;
    if (!aligned16(conv_state_in) || !aligned16(conv_state_out) || !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    if (N == 0 && conv_state_out == nullptr) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    const __nv_bfloat16 *xb[3];
    __nv_bfloat16 *yb[3];
    for (int i = 0; i < 3; ++i) {
        xb[i] = static_cast<const __nv_bfloat16 *>(xs[i]);
        yb[i] = static_cast<__nv_bfloat16 *>(ys[i]);
    }
    return from_cuda(kda::launch_short_conv(
        xb, ws, yb, cu_seqlens, B, N, C, static_cast<const __nv_bfloat16 *>(conv_state_in),
        static_cast<__nv_bfloat16 *>(conv_state_out), dev->error_word,
        static_cast<cudaStream_t>(stream)));
}

kda_status kda_short_conv_qkv_step(const void *x_q, const void *x_k, const void *x_v,
                                   const float *w_q, const float *w_k, const float *w_v,
                                   void *conv_state_pool, const int32_t *state_indices,
                                   int num_slots, int B, int C,
                                   void *q, void *k, void *v, void *stream) {
    if (B < 0 || B > 65535 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (state_indices == nullptr && num_slots < B) return KDA_ERR_INVALID_ARG;
    if (C < 128 || C % 128 != 0) return KDA_ERR_UNSUPPORTED_SHAPE;
    const void *xs[3] = {x_q, x_k, x_v};
    const float *ws[3] = {w_q, w_k, w_v};
    void *ys[3] = {q, k, v};
    if (B > 0) {
        for (int i = 0; i < 3; ++i)
            if (xs[i] == nullptr || ws[i] == nullptr || ys[i] == nullptr) return KDA_ERR_INVALID_ARG;
        if (conv_state_pool == nullptr) return KDA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < 3; ++i)
        if (!aligned16(xs[i]) || !aligned16(ws[i]) || !aligned16(ys[i])) return KDA_ERR_MISALIGNED;
    if (!aligned16(conv_state_pool) || !aligned16(state_indices)) return KDA_ERR_MISALIGNED;
    if (B == 0) return KDA_OK;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    const __nv_bfloat16 *xb[3];
    __nv_bfloat16 *yb[3];
    for (int i = 0; i < 3; ++i) {
        xb[i] = static_cast<const __nv_bfloat16 *>(xs[i]);
        yb[i] = static_cast<__nv_bfloat16 *>(ys[i]);
    }
    return from_cuda(kda::launch_short_conv_step(
        xb, ws, yb, static_cast<__nv_bfloat16 *>(conv_state_pool), state_indices, num_slots, B, C,
        dev->error_word, static_cast<cudaStream_t>(stream)));
}

size_t kda_recurrent_backward_workspace_size(int64_t N, int B, int H, int K, int V) {
    if (N < 0 || B < 1 || H < 1 || K != 128 || V != 128) return 0;
    return kda::backward_workspace_bytes(N, B, H, kda::backward_ctas(B, H, kda::kBackwardMaxCtas));
}

kda_status kda_recurrent_backward(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const int32_t *cu_seqlens, int B, int64_t N,
                                  int H, int K, int V, float scale, const float *initial_state,
                                  const void *dO, kda_dtype dO_dtype, const float *dS_final,
                                  float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                  float *dS0, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (N < 0 || B < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(dO_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (cu_seqlens == nullptr && B != 1) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || dO == nullptr || dq == nullptr || dk == nullptr ||
                  dv == nullptr || dg == nullptr || dbeta == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
        !aligned16(dbeta) || !aligned16(initial_state) || !aligned16(dS_final) ||
        !aligned16(dS0) || !aligned16(workspace) || !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    const size_t need = kda_recurrent_backward_workspace_size(N, B, H, K, V);
    if (workspace_bytes < need || workspace == nullptr) return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    const int ctas = kda::backward_ctas(B, H, dev->num_sms < kda::kBackwardMaxCtas
                                                  ? dev->num_sms : kda::kBackwardMaxCtas);
    return from_cuda(kda::launch_backward(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, B, N, H, scale, initial_state,
        dO, dO_dtype == KDA_BF16, dS_final, dq, dk, dv, dg, dbeta, dS0, workspace, ctas,
        dev->error_word, static_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_backward_workspace_size(int64_t N, int B, int H, int K, int V) {
    if (N < 0 || B < 1 || H < 1 || K != 128 || V != 128) return 0;
    const int64_t chains = static_cast<int64_t>(B) * H;
    const int ctas = static_cast<int>(chains < kda::kChunkBwdMaxCtas ? chains : kda::kChunkBwdMaxCtas);
    return kda::chunk_bwd_workspace_bytes(N, B, H, ctas);
}

kda_status kda_chunk_backward(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const int32_t *cu_seqlens, int B, int64_t N,
                              int H, int K, int V, float scale, const float *initial_state,
                              const void *dO, kda_dtype dO_dtype, const float *dS_final,
                              float *dq, float *dk, float *dv, float *dg, float *dbeta,
                              float *dS0, void *workspace, size_t workspace_bytes, void *stream) {
    if (N < 0 || B < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(dO_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (cu_seqlens == nullptr && B != 1) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || dO == nullptr || dq == nullptr || dk == nullptr ||
                  dv == nullptr || dg == nullptr || dbeta == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
        !aligned16(dbeta) || !aligned16(initial_state) || !aligned16(dS_final) ||
        !aligned16(dS0) || !aligned16(workspace) || !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    const size_t need = kda_chunk_backward_workspace_size(N, B, H, K, V);
    if (workspace_bytes < need || workspace == nullptr) return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    const int64_t chains = static_cast<int64_t>(B) * H;
    int ctas = dev->num_sms < kda::kChunkBwdMaxCtas ? dev->num_sms : kda::kChunkBwdMaxCtas;
    if (chains < ctas) ctas = static_cast<int>(chains);
    return from_cuda(kda::launch_chunk_backward(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, B, N, H, scale, initial_state,
        dO, dO_dtype == KDA_BF16, dS_final, dq, dk, dv, dg, dbeta, dS0, workspace, ctas,
        dev->error_word, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_checkpoints_size(int64_t N, int B, int H, int K, int V) {
    if (N < 0 || B < 1 || H < 1 || K != 128 || V != 128) return 0;
    return kda::chunk_checkpoints_bytes(N, B, H);
}

kda_status kda_chunk_prefill_checkpointed(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const int32_t *cu_seqlens, int B, int64_t N, int H,
                                          int K, int V, float scale, const float *initial_state,
                                          float *final_state, void *o, kda_dtype o_dtype,
                                          void *checkpoints, size_t checkpoints_bytes,
                                          void *workspace, size_t workspace_bytes, void *stream) {
    kda_status st = check_prefill_args(q, k, v, g, beta, cu_seqlens, B, N, H, K, V, initial_state,
                                       final_state, o, o_dtype);
    if (st != KDA_OK) return st;
    if (!aligned16(workspace) || !aligned16(checkpoints)) return KDA_ERR_MISALIGNED;
    const size_t need = kda::prefill_workspace_bytes(N, B, H);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    if (checkpoints == nullptr || checkpoints_bytes < kda::chunk_checkpoints_bytes(N, B, H))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    st = current_device(&dev);
    if (st != KDA_OK) return st;
    uint8_t *cp = static_cast<uint8_t *>(checkpoints);
    return from_cuda(kda::launch_prefill_checkpointed(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, B, N, H, scale, initial_state,
        final_state, o, o_dtype == KDA_BF16,
        reinterpret_cast<float *>(cp + kda::chunk_checkpoint_flags_bytes(B, H)),
        reinterpret_cast<int *>(cp), workspace, dev->error_word, dev->num_sms,
        static_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_backward_checkpointed_workspace_size(int64_t N, int B, int H, int K, int V) {
    if (N < 0 || B < 1 || H < 1 || K != 128 || V != 128) return 0;
    const int64_t chains = static_cast<int64_t>(B) * H;
    const int ctas = static_cast<int>(chains < kda::kChunkBwdMaxCtas ? chains : kda::kChunkBwdMaxCtas);
    return kda::chunk_bwd_from_checkpoints_workspace_bytes(ctas);
}

kda_status kda_chunk_backward_checkpointed(const void *q, const void *k, const void *v,
                                           const float *g, const float *beta,
                                           const int32_t *cu_seqlens, int B, int64_t N, int H,
                                           int K, int V, float scale, const void *checkpoints,
                                           size_t checkpoints_bytes, const void *dO,
                                           kda_dtype dO_dtype, const float *dS_final, float *dq,
                                           float *dk, float *dv, float *dg, float *dbeta,
                                           float *dS0, void *workspace, size_t workspace_bytes,
                                           void *stream) {
    if (N < 0 || B < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!valid_dtype(dO_dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (cu_seqlens == nullptr && B != 1) return KDA_ERR_INVALID_ARG;
    if (N > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr ||
                  beta == nullptr || dO == nullptr || dq == nullptr || dk == nullptr ||
                  dv == nullptr || dg == nullptr || dbeta == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
        !aligned16(dbeta) || !aligned16(checkpoints) || !aligned16(dS_final) ||
        !aligned16(dS0) || !aligned16(workspace) || !aligned16(cu_seqlens))
        return KDA_ERR_MISALIGNED;
    if (checkpoints == nullptr || checkpoints_bytes < kda::chunk_checkpoints_bytes(N, B, H))
        return KDA_ERR_WORKSPACE_TOO_SMALL;
    const size_t need = kda_chunk_backward_checkpointed_workspace_size(N, B, H, K, V);
    if (workspace_bytes < need || workspace == nullptr) return KDA_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    const int64_t chains = static_cast<int64_t>(B) * H;
    int ctas = dev->num_sms < kda::kChunkBwdMaxCtas ? dev->num_sms : kda::kChunkBwdMaxCtas;
    if (chains < ctas) ctas = static_cast<int>(chains);
    return from_cuda(kda::launch_chunk_backward_from_checkpoints(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, B, N, H, scale, checkpoints,
        dO, dO_dtype == KDA_BF16, dS_final, dq, dk, dv, dg, dbeta, dS0, workspace, ctas,
        dev->error_word, static_cast<cudaStream_t>(stream)));
}

kda_status kda_debug_check_gate_division(uint64_t *mismatches, void *stream) {
    if (mismatches == nullptr) return KDA_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    unsigned long long n = 0;
    st = from_cuda(kda::check_gate_division(&n, dev->num_sms, static_cast<cudaStream_t>(stream)));
    if (st != KDA_OK) return st;
    *mismatches = static_cast<uint64_t>(n);
    return KDA_OK;
}

kda_status kda_debug_set_wait_limit(int64_t copy_polls, int64_t product_polls) {
    kda::set_prefill_wait_polls(copy_polls, product_polls);
    return KDA_OK;
}

kda_status kda_get_last_device_error(void *stream) {
    DeviceInfo *dev = nullptr;
    kda_status st = current_device(&dev);
    if (st != KDA_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word)) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero)) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
    }
    return static_cast<kda_status>(word);
}

}  // extern "C"
