// claims.cu -- the counters through which the CTAs of one pipeline launch claim their
// work units (pipeline.cuh), host side.
//
// A launch that hands out its units dynamically needs a pair of device words (units
// claimed, CTAs done) that start at zero and that no other launch touches while it
// runs.  Each device has a ring of kClaimSlots such pairs.  A launch takes a slot whose
// previous launch is known to be complete -- an event recorded on that launch's stream
// right after it has completed -- and records the slot's event after its own launch.
// The kernel leaves the pair at zero when its last CTA is done with claiming (the last
// producer to count itself out clears both words), so no clearing launch is queued.
// A slot is therefore never shared by two launches that may overlap, whatever streams
// and threads they come from.  When no slot is free, under stream capture, or when the
// ring cannot be set up, the launch gets no slot and splits its units statically.
//
// The ring holds 1024 pairs: a host that queues a long run of steps ahead of the GPU
// (50 steps of the 4-block Llama, three claiming launches each, are queued within about
// a millisecond) must not run out of pairs, or its later launches fall back to the static
// split (measured on GB300 with a 64-pair ring: those steps 4 % slower, launch times
// spread by 4 %).  Slots are taken in turn, so the one at the cursor is the oldest; a
// launch looks at no more than kClaimProbe of them.
#include <cstdint>
#include <mutex>

#include "staged.hpp"

namespace fsdp {
namespace {

constexpr int kClaimSlots = 1024;
constexpr int kClaimProbe = 16;
constexpr int kClaimDevices = 64;

struct Ring {
    bool ready = false, failed = false;
    unsigned int* dev = nullptr;          // kClaimSlots pairs (units claimed, CTAs done)
    cudaEvent_t ev[kClaimSlots] = {};
    bool recorded[kClaimSlots] = {};      // ev[k] follows the slot's last launch
    bool held[kClaimSlots] = {};          // taken by a launch not yet recorded
    int next = 0;
};

std::mutex g_claim_mu;
Ring g_rings[kClaimDevices];

// The device's ring, set up on first use (one allocation, zeroed, and the events);
// nullptr when that failed.  Caller holds g_claim_mu.
Ring* ring_of(int dev) {
    Ring& r = g_rings[dev];
    if (r.failed) return nullptr;
    if (r.ready) return &r;
    const size_t bytes = size_t(kClaimSlots) * 2 * sizeof(unsigned int);
    bool ok = cudaMalloc(&r.dev, bytes) == cudaSuccess && cudaMemset(r.dev, 0, bytes) == cudaSuccess;
    for (int k = 0; ok && k < kClaimSlots; ++k)
        ok = cudaEventCreateWithFlags(&r.ev[k], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();               // leave no error behind: the launches run statically
        r.failed = true;
        return nullptr;
    }
    r.ready = true;
    return &r;
}

}  // namespace

unsigned int* claim_acquire(cudaStream_t st, int* slot, int* dev_out) {
    *slot = -1;
    *dev_out = -1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kClaimDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_claim_mu);
    Ring* r = ring_of(dev);
    if (!r) return nullptr;
    for (int i = 0; i < kClaimProbe; ++i) {
        const int k = (r->next + i) % kClaimSlots;
        if (r->held[k]) continue;
        if (r->recorded[k]) {
            const cudaError_t q = cudaEventQuery(r->ev[k]);
            if (q != cudaSuccess) {       // still running (or an error: not provably free)
                if (q != cudaErrorNotReady) cudaGetLastError();
                continue;
            }
        }
        r->held[k] = true;
        r->next = (k + 1) % kClaimSlots;
        *slot = k;
        *dev_out = dev;
        return r->dev + 2 * k;
    }
    return nullptr;
}

void claim_release(int slot, int dev, cudaStream_t st, bool launched) {
    if (slot < 0 || dev < 0 || dev >= kClaimDevices) return;
    std::lock_guard<std::mutex> lk(g_claim_mu);
    Ring& r = g_rings[dev];
    if (launched) {
        if (cudaEventRecord(r.ev[slot], st) != cudaSuccess) {
            cudaGetLastError();
            return;                       // not provably free again: the slot stays held
        }
        r.recorded[slot] = true;
    }
    r.held[slot] = false;
}

}  // namespace fsdp
