// The C ABI (include/gdn.h): argument validation, status codes, the per-device
// error word, tensor-map encoding, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gdn {

constexpr int kMaxDevicesHost = 64;

// One word per device, set by kernels whose bounded waits give up.
__device__ unsigned g_error_word;

namespace {

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

unsigned *error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned *>(ptr);
    }
    return g_err_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A tensor pointer is acceptable if 16-byte aligned and, when the tensor has
// elements, not null.
bool ok_ptr(const void *p, size_t elems) { return aligned16(p) && (elems == 0 || p != nullptr); }

bool supported_d(int d) { return d == 32 || d == 64 || d == 128; }

gdn_status check_dims(const gdn_dims *d, Sizes *s) {
    if (d == nullptr) return GDN_ERR_INVALID_ARG;
    if (d->B < 0 || d->T < 0 || d->Hk <= 0 || d->Hv <= 0 || d->Dk <= 0 || d->Dv <= 0 || d->K <= 0)
        return GDN_ERR_INVALID_ARG;
    if (d->Hv % d->Hk != 0) return GDN_ERR_INVALID_ARG;
    if (!(d->eps_qk >= 0.0f)) return GDN_ERR_INVALID_ARG;
    if (!supported_d(d->Dk) || !supported_d(d->Dv) || d->K < 2 || d->K > 4) return GDN_ERR_UNSUPPORTED;
    if ((long long)d->B > 65535) return GDN_ERR_UNSUPPORTED;
    const long long C = 2LL * d->Hk * d->Dk + (long long)d->Hv * d->Dv;
    if (C > (1LL << 30) || (long long)d->Hv * d->Dv > 65535LL * 128) return GDN_ERR_UNSUPPORTED;
    *s = Sizes{d->B, d->T, d->Hk, d->Hv, d->Dk, d->Dv, d->K, d->eps_qk};
    return GDN_OK;
}

gdn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    return e == cudaErrorNotSupported ? GDN_ERR_UNSUPPORTED : GDN_ERR_CUDA;
}

}  // namespace

int num_sms() {
    const int dev = current_device();
    if (dev < 0) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool encode_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, uint64_t d2,
                    uint64_t d1, uint64_t d0, uint32_t box1, uint32_t box0) {
    const auto fn = tmap_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * (cuuint64_t)elem_bytes, d1 * d0 * (cuuint64_t)elem_bytes};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, int rank,
                 const uint64_t *dims, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    const auto fn = tmap_encoder();
    if (fn == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t gdims[5], strides[4];
    cuuint32_t gbox[5], estr[5];
    cuuint64_t pitch = (cuuint64_t)elem_bytes;
    for (int i = 0; i < rank; ++i) {
        gdims[i] = dims[i];
        gbox[i] = box[i];
        estr[i] = 1;
        if (i > 0) strides[i - 1] = pitch;
        pitch *= dims[i];
    }
    return fn(map, dtype, (cuuint32_t)rank, const_cast<void *>(base), gdims, strides, gbox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, uint64_t rows,
                    uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    const auto fn = tmap_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// gdn_prefill and gdn_prefill_gated: z == nullptr gives y, else the gated norm.
static gdn_status prefill_impl(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const float *g, const float *beta, const float *state_in, float *state_out,
                               const uint8_t *mask, uint16_t *y, const uint16_t *z, const float *norm_w,
                               float norm_eps, int chunk, void *workspace, size_t ws_bytes, gdn_stream stream) {
    Sizes s;
    gdn_status st = check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (chunk != 0 && chunk != 64) return GDN_ERR_UNSUPPORTED;
    const size_t BT = (size_t)s.B * s.T;
    const size_t nstate = (size_t)s.B * s.Hv * s.Dv * s.Dk;
    if (!ok_ptr(q, BT) || !ok_ptr(k, BT) || !ok_ptr(v, BT) || !ok_ptr(g, BT) || !ok_ptr(beta, BT) ||
        !ok_ptr(state_in, 0) || !ok_ptr(state_out, nstate) || !ok_ptr(mask, 0) || !ok_ptr(y, BT))
        return GDN_ERR_INVALID_ARG;
    if (z != nullptr && (!ok_ptr(norm_w, 1) || !(norm_eps >= 0.0f))) return GDN_ERR_INVALID_ARG;
    if (workspace != nullptr && (ws_bytes < row_order_workspace(s) || !aligned16(workspace)))
        return GDN_ERR_INVALID_ARG;
    if (s.B == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    if (s.T == 0) {
        if (state_in == nullptr) return from_cuda(cudaMemsetAsync(state_out, 0, nstate * sizeof(float), cs));
        if (state_in == state_out) return GDN_OK;
        return from_cuda(
            cudaMemcpyAsync(state_out, state_in, nstate * sizeof(float), cudaMemcpyDeviceToDevice, cs));
    }
    // rows of a masked batch longest first (scheduling only; results identical)
    const int *order = nullptr;
    if (mask != nullptr && workspace != nullptr && s.B > 1) {
        cudaError_t e = launch_row_order(s, mask, workspace, cs);
        if (e != cudaSuccess) return from_cuda(e);
        order = static_cast<const int *>(workspace);
    }
    if (chunk == 0) {
        // the sequential kernel spreads a head's rows over several CTAs: y goes
        // to the output buffer and the gated norm runs over it in place
        cudaError_t e = launch_prefill_seq(s, q, k, v, g, beta, state_in, state_out, mask, order, y,
                                           error_word(), cs);
        if (e == cudaSuccess && z != nullptr) e = launch_rmsnorm_gated(s, y, z, norm_w, norm_eps, y, cs);
        return from_cuda(e);
    }
    // Chunked form with few heads and a workspace of the full size: two passes
    // (the state-independent work of every chunk spread over the GPU first)
    const size_t ws_order = row_order_workspace(s);
    if (prefill_two_pass_pays(s) && workspace != nullptr &&
        ws_bytes >= ws_order + prefill_two_pass_workspace(s)) {
        cudaError_t e = launch_prefill_two_pass(s, q, k, v, g, beta, state_in, state_out, mask, order, y,
                                                static_cast<char *>(workspace) + ws_order, error_word(), cs);
        if (e == cudaSuccess && z != nullptr) e = launch_rmsnorm_gated(s, y, z, norm_w, norm_eps, y, cs);
        return from_cuda(e);
    }
    // Chunked form: the norm in the kernel's epilogue when there are at least
    // as many heads as SMs.  With fewer, each head's chain of chunks is the
    // critical path and the epilogue lengthens every link of it, while a
    // separate norm kernel spreads over the whole GPU (measured at B = 1,
    // Hv = 32, T = 8192: 1.52 ms fused against 1.41 ms; at B = 8, Hv = 64,
    // ragged T = 16384: 4.54 ms fused against 5.20 ms).
    const bool fuse = z != nullptr && (long)s.B * s.Hv >= num_sms();
    cudaError_t e = launch_prefill_chunked(s, q, k, v, g, beta, state_in, state_out, mask, order, y,
                                           fuse ? z : nullptr, norm_w, norm_eps, error_word(), cs);
    if (e == cudaSuccess && z != nullptr && !fuse) e = launch_rmsnorm_gated(s, y, z, norm_w, norm_eps, y, cs);
    return from_cuda(e);
}

}  // namespace gdn

using gdn::ok_ptr;

extern "C" {

int gdn_abi_version(void) { return 1; }

const char *gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument (null/misaligned pointer or bad size)";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: size outside the supported set";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "GDN_ERR_UNKNOWN";
    }
}

gdn_status gdn_conv_update(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                           uint16_t *conv_state, const uint8_t *mask, uint16_t *q, uint16_t *k, uint16_t *v,
                           gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    const size_t BT = (size_t)s.B * s.T;
    if (!ok_ptr(qkv, BT * s.C()) || !ok_ptr(conv_w, BT) || !ok_ptr(conv_state, 0) || !ok_ptr(mask, 0) ||
        !ok_ptr(q, BT) || !ok_ptr(k, BT) || !ok_ptr(v, BT))
        return GDN_ERR_INVALID_ARG;
    if (BT == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_conv_update(s, qkv, conv_w, conv_state, mask, q, k, v, gdn::error_word(),
                                                  (cudaStream_t)stream));
}

gdn_status gdn_gating(const gdn_dims *dims, const uint16_t *a, const uint16_t *b, const float *A_log,
                      const float *dt_bias, float *g, float *beta, gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    const size_t n = (size_t)s.B * s.T * s.Hv;
    if (!ok_ptr(a, n) || !ok_ptr(b, n) || !ok_ptr(A_log, n) || !ok_ptr(dt_bias, n) || !ok_ptr(g, n) ||
        !ok_ptr(beta, n))
        return GDN_ERR_INVALID_ARG;
    if (n == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_gating(s, a, b, A_log, dt_bias, g, beta, (cudaStream_t)stream));
}

gdn_status gdn_recurrent_decode(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                                uint16_t *conv_state, const uint16_t *a, const uint16_t *b, const float *A_log,
                                const float *dt_bias, float *state, const uint8_t *row_mask, uint16_t *y,
                                gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (s.T != 1) return GDN_ERR_INVALID_ARG;
    if (s.Hv / s.Hk > 16) return GDN_ERR_UNSUPPORTED;
    const size_t B = (size_t)s.B;
    if (!ok_ptr(qkv, B) || !ok_ptr(conv_w, B) || !ok_ptr(conv_state, B) || !ok_ptr(a, B) || !ok_ptr(b, B) ||
        !ok_ptr(A_log, B) || !ok_ptr(dt_bias, B) || !ok_ptr(state, B) || !ok_ptr(row_mask, 0) || !ok_ptr(y, B))
        return GDN_ERR_INVALID_ARG;
    if (B == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_decode(s, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, y,
                                             nullptr, nullptr, 0.0f, gdn::error_word(), (cudaStream_t)stream));
}

namespace {

// Staging slots of gdn_recurrent_decode_host_steps: step i uses slot i %
// kHostSlots, so inputs run up to kHostSlots - 1 steps ahead of the kernels
// and a short stall of the copy path is absorbed.
constexpr int kHostSlots = 4;

// One staging slot of gdn_recurrent_decode_host_steps: byte offsets of qkv,
// a, b and y (each 256-byte aligned) and the slot size.
struct HostSlot {
    size_t qkv, a, b, y, bytes;
};

// The copy streams and events of gdn_recurrent_decode_host_steps, created on
// a device's first call and kept for the life of the process (creating them
// on every call cost about as much host time as a few decode steps).  A
// call holds the device's mutex while it enqueues, so calls from several
// host threads do not interleave their records and waits on the shared
// events.
struct HostLoop {
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t start = nullptr, in[kHostSlots] = {}, done[kHostSlots] = {}, out[kHostSlots] = {};
    std::mutex mu;
    bool ready = false;
};
HostLoop g_host_loop[gdn::kMaxDevicesHost];

cudaError_t host_loop_setup(HostLoop &h) {
    if (h.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&h.cin, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.cout, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming);
    for (int k = 0; k < kHostSlots && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&h.in[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.done[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.out[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        // release what was made; the next call tries again
        for (int k = 0; k < kHostSlots; ++k) {
            if (h.in[k]) cudaEventDestroy(h.in[k]);
            if (h.done[k]) cudaEventDestroy(h.done[k]);
            if (h.out[k]) cudaEventDestroy(h.out[k]);
            h.in[k] = h.done[k] = h.out[k] = nullptr;
        }
        if (h.start) cudaEventDestroy(h.start);
        if (h.cin) cudaStreamDestroy(h.cin);
        if (h.cout) cudaStreamDestroy(h.cout);
        h.start = nullptr;
        h.cin = h.cout = nullptr;
        return e;
    }
    h.ready = true;
    return cudaSuccess;
}

HostSlot host_slot(const gdn::Sizes &s) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    HostSlot h;
    h.qkv = 0;
    h.a = up((size_t)s.B * s.C() * 2);
    h.b = h.a + up((size_t)s.B * s.Hv * 2);
    h.y = h.b + up((size_t)s.B * s.Hv * 2);
    h.bytes = h.y + up((size_t)s.B * s.Hv * s.Dv * 2);
    return h;
}

}  // namespace

size_t gdn_decode_host_staging_size(const gdn_dims *dims) {
    gdn::Sizes s;
    if (gdn::check_dims(dims, &s) != GDN_OK || s.T != 1) return 0;
    return kHostSlots * host_slot(s).bytes;
}

gdn_status gdn_recurrent_decode_host_steps(const gdn_dims *dims, int n_steps, const uint16_t *qkv_h,
                                           const uint16_t *a_h, const uint16_t *b_h, uint16_t *y_h,
                                           const uint16_t *conv_w, uint16_t *conv_state, const float *A_log,
                                           const float *dt_bias, float *state, const uint8_t *row_mask,
                                           void *staging, size_t staging_bytes, gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (s.T != 1 || n_steps < 0) return GDN_ERR_INVALID_ARG;
    if (s.Hv / s.Hk > 16) return GDN_ERR_UNSUPPORTED;
    const size_t B = (size_t)s.B;
    if (n_steps == 0 || B == 0) return GDN_OK;
    if (qkv_h == nullptr || a_h == nullptr || b_h == nullptr || y_h == nullptr) return GDN_ERR_INVALID_ARG;
    if (!ok_ptr(conv_w, B) || !ok_ptr(conv_state, B) || !ok_ptr(A_log, B) || !ok_ptr(dt_bias, B) ||
        !ok_ptr(state, B) || !ok_ptr(row_mask, 0) || !ok_ptr(staging, B))
        return GDN_ERR_INVALID_ARG;
    const HostSlot h = host_slot(s);
    if (staging_bytes < kHostSlots * h.bytes) return GDN_ERR_INVALID_ARG;
    const size_t nq = B * s.C(), na = B * s.Hv, ny = B * s.Hv * s.Dv;   // elements per step

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gdn::kMaxDevicesHost) return GDN_ERR_CUDA;
    HostLoop &hl = g_host_loop[dev];
    std::lock_guard<std::mutex> lk(hl.mu);
    cudaError_t e = host_loop_setup(hl);
    if (e != cudaSuccess) return gdn::from_cuda(e);
    cudaStream_t main = (cudaStream_t)stream, cin = hl.cin, cout = hl.cout;
    cudaEvent_t ev_start = hl.start, *ev_in = hl.in, *ev_done = hl.done, *ev_out = hl.out;
    // the copy streams start after everything already on `stream`; every slot
    // starts free (its "done" and "out" events complete at that point)
    if (e == cudaSuccess) e = cudaEventRecord(ev_start, main);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cin, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cout, ev_start, 0);
    for (int k = 0; k < kHostSlots && e == cudaSuccess; ++k) {
        e = cudaEventRecord(ev_done[k], main);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[k], main);
    }
    for (int i = 0; i < n_steps && e == cudaSuccess; ++i) {
        const int k = i % kHostSlots;
        char *slot = static_cast<char *>(staging) + (size_t)k * h.bytes;
        uint16_t *qkv_d = reinterpret_cast<uint16_t *>(slot + h.qkv);
        uint16_t *a_d = reinterpret_cast<uint16_t *>(slot + h.a);
        uint16_t *b_d = reinterpret_cast<uint16_t *>(slot + h.b);
        uint16_t *y_d = reinterpret_cast<uint16_t *>(slot + h.y);
        // step i's inputs, once the slot's previous step has finished reading it
        e = cudaStreamWaitEvent(cin, ev_done[k], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(qkv_d, qkv_h + (size_t)i * nq, nq * 2, cudaMemcpyHostToDevice, cin);
        if (e == cudaSuccess) e = cudaMemcpyAsync(a_d, a_h + (size_t)i * na, na * 2, cudaMemcpyHostToDevice, cin);
        if (e == cudaSuccess) e = cudaMemcpyAsync(b_d, b_h + (size_t)i * na, na * 2, cudaMemcpyHostToDevice, cin);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[k], cin);
        // the step, once its inputs are in and the slot's previous y has left it
        if (e == cudaSuccess) e = cudaStreamWaitEvent(main, ev_in[k], 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(main, ev_out[k], 0);
        if (e == cudaSuccess)
            e = gdn::launch_decode(s, qkv_d, conv_w, conv_state, a_d, b_d, A_log, dt_bias, state, row_mask, y_d,
                                   nullptr, nullptr, 0.0f, gdn::error_word(), main);
        if (e == cudaSuccess) e = cudaEventRecord(ev_done[k], main);
        // step i's y back to the host
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cout, ev_done[k], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(y_h + (size_t)i * ny, y_d, ny * 2, cudaMemcpyDeviceToHost, cout);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[k], cout);
    }
    // `stream` completes after the last y has arrived
    for (int k = 0; k < kHostSlots && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(main, ev_out[k], 0);
    return gdn::from_cuda(e);
}

gdn_status gdn_recurrent_decode_gated(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                                      uint16_t *conv_state, const uint16_t *a, const uint16_t *b,
                                      const float *A_log, const float *dt_bias, float *state,
                                      const uint8_t *row_mask, const uint16_t *z, const float *norm_w,
                                      float norm_eps, uint16_t *out, gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (s.T != 1) return GDN_ERR_INVALID_ARG;
    if (s.Hv / s.Hk > 16) return GDN_ERR_UNSUPPORTED;
    if (!(norm_eps >= 0.0f)) return GDN_ERR_INVALID_ARG;
    const size_t B = (size_t)s.B;
    if (!ok_ptr(qkv, B) || !ok_ptr(conv_w, B) || !ok_ptr(conv_state, B) || !ok_ptr(a, B) || !ok_ptr(b, B) ||
        !ok_ptr(A_log, B) || !ok_ptr(dt_bias, B) || !ok_ptr(state, B) || !ok_ptr(row_mask, 0) || !ok_ptr(z, B) ||
        !ok_ptr(norm_w, B) || !ok_ptr(out, B))
        return GDN_ERR_INVALID_ARG;
    if (B == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_decode(s, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, out,
                                             z, norm_w, norm_eps, gdn::error_word(), (cudaStream_t)stream));
}

gdn_status gdn_decode_window(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                             uint16_t *conv_state, const uint16_t *a, const uint16_t *b, const float *A_log,
                             const float *dt_bias, float *state, const int32_t *keep, uint16_t *y,
                             gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (s.T < 1 || s.T > 8) return GDN_ERR_UNSUPPORTED;
    if (s.Hv / s.Hk > 16) return GDN_ERR_UNSUPPORTED;
    const size_t B = (size_t)s.B;
    if (!ok_ptr(qkv, B) || !ok_ptr(conv_w, B) || !ok_ptr(conv_state, B) || !ok_ptr(a, B) || !ok_ptr(b, B) ||
        !ok_ptr(A_log, B) || !ok_ptr(dt_bias, B) || !ok_ptr(state, B) || !ok_ptr(keep, 0) || !ok_ptr(y, B))
        return GDN_ERR_INVALID_ARG;
    if (B == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_decode_window(s, qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep,
                                                    y, gdn::error_word(), (cudaStream_t)stream));
}

size_t gdn_prefill_workspace_size(const gdn_dims *dims, int chunk) {
    gdn::Sizes s;
    if (gdn::check_dims(dims, &s) != GDN_OK) return 0;
    if (chunk != 0 && chunk != 64) return 0;
    size_t n = gdn::row_order_workspace(s);
    if (chunk == 64 && s.B > 0 && s.T > 0 && gdn::prefill_two_pass_pays(s))
        n += gdn::prefill_two_pass_workspace(s);
    return n;
}

gdn_status gdn_prefill(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *g, const float *beta, const float *state_in, float *state_out,
                       const uint8_t *mask, uint16_t *y, int chunk, void *workspace, size_t ws_bytes,
                       gdn_stream stream) {
    return gdn::prefill_impl(dims, q, k, v, g, beta, state_in, state_out, mask, y, nullptr, nullptr, 0.0f, chunk,
                        workspace, ws_bytes, stream);
}

gdn_status gdn_prefill_gated(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const float *g, const float *beta, const float *state_in, float *state_out,
                             const uint8_t *mask, const uint16_t *z, const float *norm_w, float norm_eps,
                             uint16_t *out, int chunk, void *workspace, size_t ws_bytes, gdn_stream stream) {
    const size_t BT = dims == nullptr ? 0 : (size_t)(dims->B > 0 ? dims->B : 0) * (size_t)(dims->T > 0 ? dims->T : 0);
    if (!gdn::ok_ptr(z, BT) || z == nullptr) return GDN_ERR_INVALID_ARG;
    return gdn::prefill_impl(dims, q, k, v, g, beta, state_in, state_out, mask, out, z, norm_w, norm_eps, chunk,
                        workspace, ws_bytes, stream);
}

gdn_status gdn_selftest_timeout(gdn_stream stream) {
    cudaStream_t cs = (cudaStream_t)stream;
    gdn_status st = gdn_device_status(stream);       // start from a clear error word
    if (st == GDN_ERR_CUDA) return st;
    cudaError_t e = gdn::launch_selftest_timeout(gdn::error_word(), cs);
    if (e != cudaSuccess) return gdn::from_cuda(e);
    st = gdn_device_status(stream);
    if (st != GDN_ERR_TIMEOUT) return st == GDN_OK ? GDN_ERR_CUDA : st;   // the timeout went unreported
    return GDN_OK;
}

namespace gdn {

// Shared validation and dispatch of the two backward entry points.
gdn_status backward_impl(bool chunked, const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, const float *g, const float *beta, const float *state_in,
                         const uint8_t *mask, const uint16_t *dy, const float *dstate_out, float *dq, float *dk,
                         float *dv, float *dg, float *dbeta, float *dstate_in, void *workspace, size_t ws_bytes,
                         gdn_stream stream) {
    Sizes s;
    gdn_status st = check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (chunked && (s.Dk > 128 || s.Dv > 128)) return GDN_ERR_UNSUPPORTED;
    const size_t BT = (size_t)s.B * s.T;
    const size_t nstate = (size_t)s.B * s.Hv * s.Dv * s.Dk;
    if (!ok_ptr(q, BT) || !ok_ptr(k, BT) || !ok_ptr(v, BT) || !ok_ptr(g, BT) || !ok_ptr(beta, BT) ||
        !ok_ptr(state_in, 0) || !ok_ptr(mask, 0) || !ok_ptr(dy, BT) || !ok_ptr(dstate_out, 0) || !ok_ptr(dq, BT) ||
        !ok_ptr(dk, BT) || !ok_ptr(dv, BT) || !ok_ptr(dg, BT) || !ok_ptr(dbeta, BT) || !ok_ptr(dstate_in, nstate))
        return GDN_ERR_INVALID_ARG;
    if (s.B == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    if (s.T == 0) {
        // no steps: the initial state's gradient is that of the final state
        if (dstate_out == nullptr) return from_cuda(cudaMemsetAsync(dstate_in, 0, nstate * sizeof(float), cs));
        if (dstate_out == dstate_in) return GDN_OK;
        return from_cuda(
            cudaMemcpyAsync(dstate_in, dstate_out, nstate * sizeof(float), cudaMemcpyDeviceToDevice, cs));
    }
    const size_t need = chunked ? backward_chunked_workspace(s) : backward_workspace(s);
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDN_ERR_INVALID_ARG;
    if (chunked) {
        unsigned *err = error_word();
        if (err == nullptr) return GDN_ERR_CUDA;
        return from_cuda(launch_backward_chunked(s, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv,
                                                 dg, dbeta, dstate_in, workspace, err, cs));
    }
    return from_cuda(launch_backward(s, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta,
                                     dstate_in, workspace, cs));
}

}  // namespace gdn

size_t gdn_prefill_backward_workspace_size(const gdn_dims *dims) {
    gdn::Sizes s;
    if (gdn::check_dims(dims, &s) != GDN_OK) return 0;
    return gdn::backward_workspace(s);
}

gdn_status gdn_prefill_backward(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const float *g, const float *beta, const float *state_in, const uint8_t *mask,
                                const uint16_t *dy, const float *dstate_out, float *dq, float *dk, float *dv,
                                float *dg, float *dbeta, float *dstate_in, void *workspace, size_t ws_bytes,
                                gdn_stream stream) {
    return gdn::backward_impl(false, dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta,
                              dstate_in, workspace, ws_bytes, stream);
}

size_t gdn_prefill_backward_chunked_workspace_size(const gdn_dims *dims) {
    gdn::Sizes s;
    if (gdn::check_dims(dims, &s) != GDN_OK || s.Dk > 128 || s.Dv > 128) return 0;
    return gdn::backward_chunked_workspace(s);
}

gdn_status gdn_prefill_backward_chunked(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                        const uint16_t *v, const float *g, const float *beta,
                                        const float *state_in, const uint8_t *mask, const uint16_t *dy,
                                        const float *dstate_out, float *dq, float *dk, float *dv, float *dg,
                                        float *dbeta, float *dstate_in, void *workspace, size_t ws_bytes,
                                        gdn_stream stream) {
    return gdn::backward_impl(true, dims, q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta,
                              dstate_in, workspace, ws_bytes, stream);
}

gdn_status gdn_rmsnorm_gated(const gdn_dims *dims, const uint16_t *y, const uint16_t *z, const float *norm_w,
                             float norm_eps, uint16_t *out, gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    if (!(norm_eps >= 0.0f)) return GDN_ERR_INVALID_ARG;
    const size_t n = (size_t)s.B * s.T * s.Hv;
    if (!ok_ptr(y, n) || !ok_ptr(z, n) || !ok_ptr(norm_w, n) || !ok_ptr(out, n)) return GDN_ERR_INVALID_ARG;
    if (n == 0) return GDN_OK;
    return gdn::from_cuda(gdn::launch_rmsnorm_gated(s, y, z, norm_w, norm_eps, out, (cudaStream_t)stream));
}

gdn_status gdn_prefill_vec(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const float *g_vec, const float *beta, const float *state_in, float *state_out,
                           const uint8_t *mask, uint16_t *y, gdn_stream stream) {
    gdn::Sizes s;
    gdn_status st = gdn::check_dims(dims, &s);
    if (st != GDN_OK) return st;
    const size_t BT = (size_t)s.B * s.T;
    const size_t nstate = (size_t)s.B * s.Hv * s.Dv * s.Dk;
    if (!ok_ptr(q, BT) || !ok_ptr(k, BT) || !ok_ptr(v, BT) || !ok_ptr(g_vec, BT) || !ok_ptr(beta, BT) ||
        !ok_ptr(state_in, 0) || !ok_ptr(state_out, nstate) || !ok_ptr(mask, 0) || !ok_ptr(y, BT))
        return GDN_ERR_INVALID_ARG;
    if (s.B == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    if (s.T == 0) {
        if (state_in == nullptr) return gdn::from_cuda(cudaMemsetAsync(state_out, 0, nstate * sizeof(float), cs));
        if (state_in == state_out) return GDN_OK;
        return gdn::from_cuda(
            cudaMemcpyAsync(state_out, state_in, nstate * sizeof(float), cudaMemcpyDeviceToDevice, cs));
    }
    return gdn::from_cuda(gdn::launch_prefill_seq_vec(s, q, k, v, g_vec, beta, state_in, state_out, mask, y,
                                                      gdn::error_word(), cs));
}

gdn_status gdn_device_status(gdn_stream stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned *w = gdn::error_word();
    if (w == nullptr) return GDN_ERR_CUDA;
    unsigned host = 0;
    if (cudaMemcpy(&host, w, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    if (host != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
        return GDN_ERR_TIMEOUT;
    }
    return GDN_OK;
}

}  // extern "C"
