// status.cuh -- the per-device status word that kernels latch errors into.
#pragma once

namespace mqa {

// Values mirror mqa_status in include/mqa.h.
constexpr int kStatusOk = 0;
constexpr int kStatusDeviceBounds = 4;
constexpr int kStatusTimeout = 5;

// One word per device (this module's copy of the variable lives on every device that loads the
// library). The first error wins; the host reads and clears it in mqa_get_device_status().
__device__ int g_device_status = 0;

__device__ __forceinline__ void latch_status(int code) { atomicCAS(&g_device_status, 0, code); }

// Where the first wait that ran out of time gave up: {site, tile index in the CTA's range, block,
// thread}; site 0 = none. The host reads and clears it (mqa_debug_timeout_site).
enum TimeoutSite : int {
  kSiteProducerEmpty = 1,   // producer: a stage to refill
  kSiteConsumerFull = 2,    // mma.sync / CUDA-core consumers: a stage's bulk copy
  kSiteConsumerSync = 3,    // consumer-wide barrier (segment end, merge)
  kSiteMmaQ = 4,            // tcgen05 issuer: a segment's Q in shared memory
  kSiteMmaFull = 5,         // tcgen05 issuer: a stage's bulk copy
  kSiteMmaP = 6,            // tcgen05 issuer: P of a tile in tensor memory
  kSiteSoftmaxS = 7,        // tcgen05 softmax: S of a tile
  kSiteSoftmaxPv = 8,       // tcgen05 softmax: O += P V before a rescale
  kSiteSoftmaxFull = 9,     // tcgen05 softmax: a stage's bulk copy (before zeroing V rows)
  kSiteEpiloguePv = 10,     // tcgen05 epilogue: the segment's last O += P V
  kSiteDrain = 11,          // tcgen05 issuer at exit: its MMAs
  kSiteTmemDone = 12,       // tcgen05 issuer at exit: the softmax warps
  kSiteMmaPv = 13,          // tcgen05 issuer: O += P V of the tile whose S buffer it reuses
  kSiteStall = 14,          // consumers: the testing stall (a barrier nothing completes)
};
__device__ int g_timeout_site[4] = {0, 0, 0, 0};

__device__ __forceinline__ void record_timeout_site(int site, int k) {
  if (atomicCAS(&g_timeout_site[0], 0, site) == 0) {
    g_timeout_site[1] = k;
    g_timeout_site[2] = static_cast<int>(blockIdx.x);
    g_timeout_site[3] = static_cast<int>(threadIdx.x);
  }
}

}  // namespace mqa
