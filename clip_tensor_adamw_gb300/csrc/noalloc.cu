// mica_clip_grad_norms_noalloc: the joint norm and clip factor without any device allocation.
//
// mica_clip_grad_norms keeps a per-list table (tensor records, the octet prefix, chunk starts, one double per CTA
// and a ticket) in device memory it allocates once per list. Some callers cannot let a library allocate: a runtime
// that reserves its whole device-memory budget up front and treats any later cudaMalloc as a failure, a caller whose
// memory is held by another allocator so that cudaMalloc would fail, or a latency-bound loop that cannot afford
// cudaMalloc's implicit device synchronisation. This entry point runs the same norm kernel with its scratch in one
// file-scope device array instead, which every GPU that loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "host.h"
#include "mica_optim.h"
#include "plan.h"

namespace mica {
namespace {

constexpr int32_t kNoallocMaxTensors = 16384;
constexpr int32_t kNoallocMaxGrid = 1024;
constexpr size_t kRecBytes = (size_t)kNoallocMaxTensors * sizeof(TensorRec);                 // 786,432
constexpr size_t kPrefixBytes = ((size_t)(kNoallocMaxTensors + 1) * sizeof(int64_t) + 255) / 256 * 256;
constexpr size_t kFirstBytes = (size_t)kNoallocMaxGrid * sizeof(int32_t);
constexpr size_t kPartialBytes = (size_t)kNoallocMaxGrid * sizeof(double);
constexpr size_t kTableBytes = kRecBytes + kPrefixBytes + kFirstBytes;  // what each call uploads
constexpr size_t kScratchBytes = kTableBytes + kPartialBytes + 256;     // + the ticket: 930,304 bytes
static_assert(kScratchBytes == 930304, "the size the header states");

// The scratch: tensor records | octet prefix | chunk starts | per-CTA partials | ticket. Shared by every call on a
// device; each call overwrites the tables and the ticket before its kernel runs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch on each device, looked up once per device with that device current, and the host
// staging area of the tables; both are static, so a call allocates nothing on the host either. g_mu serialises the
// host side of the calls.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_addr[kMaxDevices] = {};
unsigned char g_host[kTableBytes];

mica_status noalloc_fail(mica_status s, const char* msg) {
    set_error_detail(msg);
    return s;
}

mica_status scratch_address(int device, unsigned char** out) {
    if (device < 0 || device >= kMaxDevices) return noalloc_fail(MICA_ERR_DEVICE, "device ordinal above 63");
    if (!g_addr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return noalloc_fail(MICA_ERR_CUDA, "cudaGetSymbolAddress of the norm scratch failed");
        }
        g_addr[device] = static_cast<unsigned char*>(p);
    }
    *out = g_addr[device];
    return MICA_OK;
}

}  // namespace

void noalloc_forget_addresses() {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int d = 0; d < kMaxDevices; ++d) g_addr[d] = nullptr;
}

}  // namespace mica

using namespace mica;

extern "C" mica_status mica_clip_grad_norms_noalloc(const void* const* g, const int64_t* n, int32_t T,
                                                    mica_dtype gdt, float max_norm, float inv_scale, float* d_norm,
                                                    float* d_factor, void* stream) {
    set_error_detail("");
    if (gdt != MICA_F32 && gdt != MICA_F16) return noalloc_fail(MICA_ERR_DTYPE, "gradients must be f32 or f16");
    if (!d_factor) return noalloc_fail(MICA_ERR_NULL, "d_factor is NULL");
    if (std::isnan(max_norm) || !(max_norm > 0.0f)) return noalloc_fail(MICA_ERR_HYPER, "max_norm is not > 0");
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return noalloc_fail(MICA_ERR_HYPER, "inv_scale is not finite and > 0");
    if (T < 0) return noalloc_fail(MICA_ERR_COUNT, "T is negative");
    if (T > kNoallocMaxTensors)
        return noalloc_fail(MICA_ERR_COUNT, "more than 16384 tensors: beyond this entry point's scratch");
    if (T > 0 && (!g || !n)) return noalloc_fail(MICA_ERR_NULL, "a pointer array is NULL");
    const size_t es = (gdt == MICA_F16) ? 2 : 4;
    int64_t total_octs = 0, total = 0;
    for (int32_t k = 0; k < T; ++k) {
        if (n[k] < 0 || n[k] > ((int64_t)1 << 40))
            return noalloc_fail(MICA_ERR_COUNT, "an element count is out of range");
        if (n[k] == 0) continue;
        if (!g[k]) return noalloc_fail(MICA_ERR_NULL, "a gradient with n > 0 is NULL");
        if (reinterpret_cast<uintptr_t>(g[k]) % es) return noalloc_fail(MICA_ERR_ADDRESS, "a gradient is misaligned");
        total_octs += (n[k] + kOct - 1) / kOct;
        total += n[k];
    }
    if (reinterpret_cast<uintptr_t>(d_factor) % 4 || (d_norm && reinterpret_cast<uintptr_t>(d_norm) % 4))
        return noalloc_fail(MICA_ERR_ADDRESS, "d_norm or d_factor is misaligned");

    // The tables reach the device by a copy from g_host, which the next call overwrites: a copy recorded into a
    // CUDA graph would replay whatever list was passed last. So a capturing stream is refused before any other
    // CUDA call, and the capture is left as it was.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capturing) != cudaSuccess) {
        cudaGetLastError();
        return noalloc_fail(MICA_ERR_CUDA, "cudaStreamIsCapturing failed on the stream");
    }
    if (capturing != cudaStreamCaptureStatusNone)
        return noalloc_fail(MICA_ERR_CAPTURE, "the stream is capturing a CUDA graph: this call copies its tables "
                            "from a host buffer every call reuses, so it is not recorded (nothing was queued)");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return noalloc_fail(MICA_ERR_DEVICE, "no usable CUDA device");
    }
    // every buffer: device memory of this device, and each gradient's n elements inside its allocation
    mica_status s = check_device_span(d_factor, 4, 4, dev, "d_factor", 0);
    if (s == MICA_OK && d_norm) s = check_device_span(d_norm, 4, 4, dev, "d_norm", 0);
    for (int32_t k = 0; s == MICA_OK && k < T; ++k)
        if (n[k] > 0) s = check_device_span(g[k], (size_t)n[k] * es, es, dev, "g", k);
    if (s != MICA_OK) return s;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned char* scratch = nullptr;
    if ((s = scratch_address(dev, &scratch)) != MICA_OK) return s;

    // The chunk layout the allocating entry point uses: the octet prefix of the list, equal contiguous chunks (as
    // many as the allocating entry point's, capped by this scratch), each chunk's first tensor.
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 148;
    }
    TensorRec* recs = reinterpret_cast<TensorRec*>(g_host);
    int64_t* prefix = reinterpret_cast<int64_t*>(g_host + kRecBytes);
    int32_t* first = reinterpret_cast<int32_t*>(g_host + kRecBytes + kPrefixBytes);
    prefix[0] = 0;
    int64_t nonempty = 0;
    for (int32_t k = 0; k < T; ++k) {
        const void* gp = n[k] > 0 ? g[k] : nullptr;
        recs[k] = TensorRec{nullptr, const_cast<void*>(gp), nullptr, nullptr, n[k], 0, 0};
        recs[k].vec = (reinterpret_cast<uintptr_t>(gp) % (gdt == MICA_F16 ? 16 : 32)) == 0;
        prefix[k + 1] = prefix[k] + (n[k] + kOct - 1) / kOct;
        nonempty += n[k] > 0;
    }
    int32_t grid = 1, direct = 0;
    choose_norm_shape(total_octs, nonempty, gdt == MICA_F16 ? 16 : 32, sms, kNoallocMaxGrid, &grid, &direct);
    for (int32_t b = 0; b < grid; ++b) {
        const int64_t c0 = total_octs * b / grid;
        int32_t lo = 0, hi = T;  // the last tensor whose octets start at or before c0
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) / 2;
            if (prefix[mid] <= c0) lo = mid;
            else hi = mid;
        }
        first[b] = lo;
    }

    // One copy of the tables and a zero ticket into the scratch, then the norm kernel on the same stream.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ChunkTable ct{};
    ct.recs = reinterpret_cast<const TensorRec*>(scratch);
    ct.prefix = reinterpret_cast<const int64_t*>(scratch + kRecBytes);
    ct.first = reinterpret_cast<const int32_t*>(scratch + kRecBytes + kPrefixBytes);
    ct.T = T;
    ct.grid = grid;
    ct.total_octs = total_octs;
    ct.direct = direct;
    double* d_part = reinterpret_cast<double*>(scratch + kTableBytes);
    unsigned int* d_ticket = reinterpret_cast<unsigned int*>(scratch + kTableBytes + kPartialBytes);
    cudaError_t e = cudaSuccess;
    if (T > 0) e = cudaMemcpyAsync(scratch, recs, (size_t)T * sizeof(TensorRec), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(scratch + kRecBytes, prefix, (size_t)(T + 1) * sizeof(int64_t), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(scratch + kRecBytes + kPrefixBytes, first, (size_t)grid * sizeof(int32_t),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_ticket, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return noalloc_fail(MICA_ERR_CUDA, "uploading the tables into the scratch failed");
    }
    const bool keep_l2 = total * (int64_t)es <= kKeepL2MaxGradBytes;  // as the allocating entry point chooses
    const int err = launch_norm(ct, (Dtype)gdt, inv_scale, d_part, d_ticket, max_norm, d_norm, d_factor, nullptr,
                                keep_l2, stream);
    if (err != (int)cudaSuccess) return noalloc_fail(MICA_ERR_CUDA, "the norm kernel failed to launch");
    return MICA_OK;
}
