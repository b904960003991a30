// noalloc.cu -- the stepwise ring sweep for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside another framework's fixed memory pool or allocator
// callback, plugins that are given only their input and output buffers, and
// latency-critical paths where cudaMalloc / cudaFree would synchronise the
// device.  For them the stepwise sweep's scratch (one fp32 partial O and LSE,
// plus the status word) lives in a fixed array in device memory that belongs
// to this library: kNoAllocScratchBytes on every GPU that loads this code,
// held until the process exits.
#include <mutex>

#include "ra_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr size_t kHeaderBytes = 256;                        // status word + padding
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this name is only a stand-in for the
// symbol, not a device address; host code reaches the array through the
// address cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array on the current device, looked up once
// per device (the lookup loads this code's module on that device).
ra_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return ra::set_error(RA_ERR_CUDA, "cudaGetDevice failed or device index out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return ra::set_error(RA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return RA_OK;
}

// Bytes of scratch a problem needs: the status word's 256-byte header, then
// one fp32 partial O [N, B, S, H, d] and LSE [N, B, H, S], each rounded up to
// 256 bytes; 0 when it cannot fit (the caller has checked the sizes, so the
// products below cannot overflow once a shard is known to fit).
size_t scratch_need(int64_t B, int64_t L, int64_t H, int d, int N) {
    const int64_t S = L / N;
    if (S * H * (d + 1) * 4 > (int64_t)kNoAllocScratchBytes) return 0;
    const size_t n_lse = (size_t)N * (size_t)B * (size_t)S * (size_t)H;   // <= 2^30 * 2^24
    const size_t n_o = n_lse * (size_t)d;
    const size_t need = kHeaderBytes + round256(n_o * 4) + round256(n_lse * 4);
    return need <= kNoAllocScratchBytes ? need : 0;
}

}  // namespace

extern "C" ra_status ra_ring_attn_fwd_stepwise_noalloc(const void *q, const void *k, const void *v,
                                                        float *o, float *lse, int64_t B, int64_t L,
                                                        int64_t H, int d, int N, int layout,
                                                        int causal, float scale, unsigned flags,
                                                        void *stream) {
    // the argument checks of ra_ring_attn_fwd, range limits included
    if (flags & ~RA_FLAG_INJECT_STALL) return ra::set_error(RA_ERR_INVALID_ARG, "unknown flag bits");
    if (N < 1) return ra::set_error(RA_ERR_SHAPE, "N (ring degree) must be at least 1");
    if (L < 0) return ra::set_error(RA_ERR_SHAPE, "L must be non-negative");
    if (L % N) return ra::set_error(RA_ERR_SHAPE, "N must divide L");
    if (layout == RA_ZIGZAG && (L % (2 * (int64_t)N)))
        return ra::set_error(RA_ERR_SHAPE, "zigzag needs 2N | L");
    const int64_t S = L / N;
    ra_status st = ra::check_attn_sizes(B, S, H, d, N, layout, scale);
    if (st != RA_OK) return st;
    if (B * L * H == 0) return RA_OK;
    const size_t need = scratch_need(B, L, H, d, N);
    if (need == 0)
        return ra::set_error(RA_ERR_UNSUPPORTED,
                             "problem needs more scratch than the 64 MiB array of "
                             "ra_ring_attn_fwd_stepwise_noalloc (256 + round256(B*L*H*d*4) + "
                             "round256(B*L*H*4) bytes)");
    if (!q || !k || !v || !o || !lse) return ra::set_error(RA_ERR_INVALID_ARG, "null pointer argument");
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(q) || !al(k) || !al(v) || !al(o) || !al(lse))
        return ra::set_error(RA_ERR_ALIGNMENT, "every pointer must be 16-byte aligned");

    void *base = nullptr;
    st = scratch_address(&base);
    if (st != RA_OK) return st;
    uint8_t *scratch = static_cast<uint8_t *>(base);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The status word is not cleared here: it collects the timeouts of every
    // call until ra_noalloc_check_status reads and clears it (it is zero when
    // the library is loaded).  The partials are rewritten in full by every step.
    const size_t o_part_off = kHeaderBytes;
    const size_t lse_part_off = o_part_off + round256((size_t)N * B * S * H * d * 4);

    ra::AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.status = reinterpret_cast<unsigned *>(scratch);
    a.B = B;
    a.S = S;
    a.H = H;
    a.d = d;
    a.N = N;
    a.layout = layout;
    a.causal = causal;
    a.scale = scale;
    a.ring = true;
    a.out_f32 = true;
    float *o_part = reinterpret_cast<float *>(scratch + o_part_off);
    float *lse_part = reinterpret_cast<float *>(scratch + lse_part_off);
    const char *err = nullptr;
    for (int step = 0; step < N; ++step) {
        a.ring_step = step;
        a.inject_stall = step == 0 && (flags & RA_FLAG_INJECT_STALL) != 0;
        a.o = step == 0 ? static_cast<void *>(o) : static_cast<void *>(o_part);
        a.lse = step == 0 ? lse : lse_part;
        st = ra::launch_attention(a, s, &err);
        if (st != RA_OK) return ra::set_error(st, err ? err : "attention launch failed");
        if (step > 0) {
            st = ra::launch_lse_merge(o, lse, o_part, lse_part, (int64_t)N * B, S, H, d, s, &err);
            if (st != RA_OK) return ra::set_error(st, err ? err : "merge launch failed");
        }
    }
    return RA_OK;
}

extern "C" ra_status ra_noalloc_check_status(void *stream) {
    void *base = nullptr;
    ra_status st = scratch_address(&base);
    if (st != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return ra::set_error(RA_ERR_CUDA, "cudaStreamSynchronize failed");
    if (cudaMemcpy(&word, base, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ra::set_error(RA_ERR_CUDA, "reading the scratch status word failed");
    if (word == 0) return RA_OK;
    const unsigned zero = 0;
    if (cudaMemcpy(base, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return ra::set_error(RA_ERR_CUDA, "clearing the scratch status word failed");
    if (word & ra::RA_DEV_TIMEOUT_BIT)
        return ra::set_error(RA_ERR_TIMEOUT, "a kernel of the allocation-free sweep gave up on a bounded wait");
    return ra::set_error(RA_ERR_ALIGNMENT,
                         "a kernel of the allocation-free sweep found its shared memory base unaligned");
}
