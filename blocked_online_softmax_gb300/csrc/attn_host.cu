// Host-buffer attention (attn_fwd_host): staging and copy/compute overlap.
//
// Heads are independent and contiguous in the [B, H, N, d] layout, so a large
// problem is cut into chunks of whole heads and pipelined over three internal
// streams: chunk c+1's host-to-device copies, chunk c's kernel and chunk c-1's
// device-to-host copies run at the same time. Staging memory comes from a
// library-owned stream-ordered pool that keeps its memory between calls, so a
// repeated call does not pay for a fresh device allocation each time.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace bos {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;
constexpr size_t kMinChunkBytes = (size_t)16 << 20;   // inputs per chunk below which chunking does not pay

struct HostStager {
    std::mutex mu;
    bool ready = false;
    cudaMemPool_t pool = nullptr;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[kMaxChunks] = {}, ev_comp[kMaxChunks] = {};
};

HostStager g_stagers[kMaxDevices];

bool init_stager(HostStager& hs, int dev) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&hs.pool, &props) != cudaSuccess) return false;
    uint64_t keep = UINT64_MAX;   // keep released blocks for the next call
    if (cudaMemPoolSetAttribute(hs.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&hs.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hs.s_comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hs.s_out, cudaStreamNonBlocking) != cudaSuccess)
        return false;
    if (cudaEventCreateWithFlags(&hs.ev_start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hs.ev_done, cudaEventDisableTiming) != cudaSuccess)
        return false;
    for (int c = 0; c < kMaxChunks; ++c)
        if (cudaEventCreateWithFlags(&hs.ev_in[c], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hs.ev_comp[c], cudaEventDisableTiming) != cudaSuccess)
            return false;
    hs.ready = true;
    return true;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

int host_forward(const AttnParams& p, cudaStream_t caller, int dev) {
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    HostStager& hs = g_stagers[dev];
    std::lock_guard<std::mutex> lk(hs.mu);   // one host-buffer call per device at a time
    if (!hs.ready && !init_stager(hs, dev)) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const int BH = p.B * p.H;
    const size_t head_t = (size_t)p.N * p.d * 2;        // bytes of one head of Q, K, V or O
    const size_t head_l = (size_t)p.N * sizeof(float);  // bytes of one head of LSE
    const size_t tbytes = head_t * BH, lbytes = head_l * BH;
    const size_t off_k = round256(tbytes), off_v = off_k + round256(tbytes), off_o = off_v + round256(tbytes),
                 off_l = off_o + round256(tbytes), total = off_l + round256(lbytes);

    // Chunks of whole heads: up to kMaxChunks, each with at least kMinChunkBytes of inputs.
    int nch = (int)((3 * tbytes) / kMinChunkBytes);
    nch = nch < 1 ? 1 : (nch > kMaxChunks ? kMaxChunks : nch);
    if (nch > BH) nch = BH;
    const int hpc = (BH + nch - 1) / nch;
    nch = (BH + hpc - 1) / hpc;

    char* base = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), total, hs.pool, caller) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const char* qh = static_cast<const char*>(p.q);
    const char* kh = static_cast<const char*>(p.k);
    const char* vh = static_cast<const char*>(p.v);
    char* oh = static_cast<char*>(p.o);
    char* lh = reinterpret_cast<char*>(p.lse);
    int rc = ATTN_OK;
    bool ok = cudaEventRecord(hs.ev_start, caller) == cudaSuccess &&
              cudaStreamWaitEvent(hs.s_in, hs.ev_start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hs.s_comp, hs.ev_start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hs.s_out, hs.ev_start, 0) == cudaSuccess;
    for (int c = 0; ok && c < nch; ++c) {
        const int h0 = c * hpc;
        const int nh = (BH - h0) < hpc ? (BH - h0) : hpc;
        const size_t ot = head_t * h0, lt = head_t * nh, ol = head_l * h0, ll = head_l * nh;
        ok = cudaMemcpyAsync(base + ot, qh + ot, lt, cudaMemcpyHostToDevice, hs.s_in) == cudaSuccess &&
             cudaMemcpyAsync(base + off_k + ot, kh + ot, lt, cudaMemcpyHostToDevice, hs.s_in) == cudaSuccess &&
             cudaMemcpyAsync(base + off_v + ot, vh + ot, lt, cudaMemcpyHostToDevice, hs.s_in) == cudaSuccess &&
             cudaEventRecord(hs.ev_in[c], hs.s_in) == cudaSuccess &&
             cudaStreamWaitEvent(hs.s_comp, hs.ev_in[c], 0) == cudaSuccess;
        if (!ok) break;
        AttnParams cp = p;
        cp.q = base + ot;
        cp.k = base + off_k + ot;
        cp.v = base + off_v + ot;
        cp.o = base + off_o + ot;
        cp.lse = reinterpret_cast<float*>(base + off_l + ol);
        cp.B = 1;
        cp.H = nh;
        set_contiguous(cp);
        rc = launch_attn_fwd(cp, hs.s_comp, dev);
        if (rc != ATTN_OK) break;
        ok = cudaEventRecord(hs.ev_comp[c], hs.s_comp) == cudaSuccess &&
             cudaStreamWaitEvent(hs.s_out, hs.ev_comp[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(oh + ot, base + off_o + ot, lt, cudaMemcpyDeviceToHost, hs.s_out) == cudaSuccess &&
             cudaMemcpyAsync(lh + ol, base + off_l + ol, ll, cudaMemcpyDeviceToHost, hs.s_out) == cudaSuccess;
    }
    if (!ok && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    // Join every internal stream back into the caller's stream, release the staging, wait.
    cudaEventRecord(hs.ev_done, hs.s_in);
    cudaStreamWaitEvent(caller, hs.ev_done, 0);
    cudaEventRecord(hs.ev_done, hs.s_comp);
    cudaStreamWaitEvent(caller, hs.ev_done, 0);
    cudaEventRecord(hs.ev_done, hs.s_out);
    cudaStreamWaitEvent(caller, hs.ev_done, 0);
    cudaFreeAsync(base, caller);
    if (cudaStreamSynchronize(caller) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    if (rc != ATTN_OK) cudaGetLastError();
    return rc;
}

}  // namespace bos
