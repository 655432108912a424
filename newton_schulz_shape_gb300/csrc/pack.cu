// Shard -> home pack and home -> shard unpack over S simulated ranks held in
// one GPU's memory (no collective).
//
// Row-shard model (Megatron-Core API page layer_sharded_a2a, route_to_ns_home /
// route_from_ns_home): rank r's buffer is its (P/S, Q) slice of every param,
// params in index order; home h's buffer holds its params complete, in
// increasing index order. A param viewed as (pre, D, post) along shard_dim
// has, on rank r, `pre` runs of (D/S)*post elements; run u lands at
// u*D*post + r*(D/S)*post of the complete param.
//
// Two-stage model (same page: a GTP_remat stage along dim 0, then a TP stage
// along partition_dim; fused into one gather here): rank r*T + t holds remat
// slice r of TP slice t; its piece is again a sequence of runs, run u landing
// at u*outer + r*mr + t*mt of the complete param.
//
// Flat model (page owner_planning, OwnerGatherPlan / OwnerScatterPlan): rank r
// holds elements [r*size/S, (r+1)*size/S) of one flat buffer; tensor i is
// [off_i, off_i + numel_i) of that buffer and goes whole to its owner.
//
// Work split: grid.y = S ranks, grid.x = fixed-size chunks of the rank
// buffer. A CTA finds the first routing entry overlapping its chunk by binary
// search, then copies every contiguous run it overlaps with 16-byte vectors
// (falling back to 4- or 2-byte words where source and destination
// alignments differ). Bit-exact.
#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "status.h"

namespace nsk {
namespace {

constexpr int PACK_THREADS = 256;

__device__ __forceinline__ void copy_run(char* dst, const char* src, long long bytes) {
  const uintptr_t ds = reinterpret_cast<uintptr_t>(dst), ss = reinterpret_cast<uintptr_t>(src);
  if (((ds ^ ss) & 15) == 0) {
    // peel to a 16-byte boundary, vector body, tail
    long long head = (16 - (ds & 15)) & 15;
    if (head > bytes) head = bytes;
    for (long long i = threadIdx.x * 2; i < head; i += 2 * blockDim.x)
      *reinterpret_cast<uint16_t*>(dst + i) = *reinterpret_cast<const uint16_t*>(src + i);
    const long long nv = (bytes - head) / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
    uint4* d4 = reinterpret_cast<uint4*>(dst + head);
    long long i = threadIdx.x;
    for (; i + 3 * blockDim.x < nv; i += 4 * blockDim.x) {
      const uint4 a = __ldcs(&s4[i]);
      const uint4 b = __ldcs(&s4[i + blockDim.x]);
      const uint4 c = __ldcs(&s4[i + 2 * blockDim.x]);
      const uint4 d = __ldcs(&s4[i + 3 * blockDim.x]);
      __stcs(&d4[i], a);
      __stcs(&d4[i + blockDim.x], b);
      __stcs(&d4[i + 2 * blockDim.x], c);
      __stcs(&d4[i + 3 * blockDim.x], d);
    }
    for (; i < nv; i += blockDim.x) __stcs(&d4[i], __ldcs(&s4[i]));
    const long long done = head + nv * 16;
    for (long long k = done + threadIdx.x * 2; k < bytes; k += 2 * blockDim.x)
      *reinterpret_cast<uint16_t*>(dst + k) = *reinterpret_cast<const uint16_t*>(src + k);
  } else if (((ds ^ ss) & 3) == 0) {
    long long head = (4 - (ds & 3)) & 3;
    if (head > bytes) head = bytes;
    for (long long i = threadIdx.x * 2; i < head; i += 2 * blockDim.x)
      *reinterpret_cast<uint16_t*>(dst + i) = *reinterpret_cast<const uint16_t*>(src + i);
    const long long nw = (bytes - head) / 4;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src + head);
    uint32_t* d = reinterpret_cast<uint32_t*>(dst + head);
    for (long long i = threadIdx.x; i < nw; i += blockDim.x) d[i] = s[i];
    for (long long k = head + nw * 4 + threadIdx.x * 2; k < bytes; k += 2 * blockDim.x)
      *reinterpret_cast<uint16_t*>(dst + k) = *reinterpret_cast<const uint16_t*>(src + k);
  } else {
    for (long long i = threadIdx.x * 2; i < bytes; i += 2 * blockDim.x)
      *reinterpret_cast<uint16_t*>(dst + i) = *reinterpret_cast<const uint16_t*>(src + i);
  }
}

__global__ void __launch_bounds__(PACK_THREADS) ns_pack_kernel(const __grid_constant__ PackParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  const int r = blockIdx.y;
  // entry coordinates: per-rank positions (row-shard, two-stage) or global
  // positions (flat); this rank's share of [g_begin, g_end) in its own buffer
  const long long base = p.flat ? static_cast<long long>(r) * p.rank_len : 0;
  const long long lo_local = max(0ll, p.g_begin - base);
  const long long hi_local = min(p.rank_len, p.g_end - base);
  const long long p0 = lo_local + static_cast<long long>(blockIdx.x) * p.chunk;
  if (p0 >= hi_local) return;
  const long long p1 = min(hi_local, p0 + p.chunk);
  const long long g0 = base + p0, g1 = base + p1;
  // first entry whose end is past g0
  long long lo = 0, hi = p.n_entries;
  while (lo < hi) {
    const long long mid = (lo + hi) / 2;
    const RouteEntry& e = p.entries[mid];
    if (e.seg_begin + e.seg_len <= g0)
      lo = mid + 1;
    else
      hi = mid;
  }
  const int eb = p.elem_bytes;
  char* rank_buf = reinterpret_cast<char*>(p.rank_ptr[r]);
  for (long long k = lo; k < p.n_entries; ++k) {
    const RouteEntry e = p.entries[k];
    if (e.seg_begin >= g1) break;
    if (e.home < 0 || e.home >= p.S) {
      if (threadIdx.x == 0) atomicOr(p.status, NS_DEV_BAD_INDEX);
      continue;
    }
    char* home_buf = reinterpret_cast<char*>(p.home_ptr[e.home]);
    const long long q0 = max(g0, e.seg_begin) - e.seg_begin;  // position inside the tensor's segment
    const long long q1 = min(g1, e.seg_begin + e.seg_len) - e.seg_begin;
    if (p.flat) {
      const long long rpos = e.seg_begin + q0 - base;
      char* rp = rank_buf + rpos * eb;
      char* hp = home_buf + (e.home_off + q0) * eb;
      if (p.to_home)
        copy_run(hp, rp, (q1 - q0) * eb);
      else
        copy_run(rp, hp, (q1 - q0) * eb);
    } else {
      const long long rbase = static_cast<long long>(r / p.T) * e.mr + static_cast<long long>(r % p.T) * e.mt;
      for (long long u = q0 / e.inner; u * e.inner < q1; ++u) {
        const long long a = max(q0, u * e.inner), b = min(q1, (u + 1) * e.inner);
        char* rp = rank_buf + (e.seg_begin + a) * eb;
        char* hp = home_buf + (e.home_off + u * e.outer + rbase + (a - u * e.inner)) * eb;
        if (p.to_home)
          copy_run(hp, rp, (b - a) * eb);
        else
          copy_run(rp, hp, (b - a) * eb);
      }
    }
  }
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, cudaStream_t st) {
  if (p.rank_len <= 0 || p.n_entries <= 0 || p.S <= 0 || p.g_end <= p.g_begin) return cudaSuccess;
  const long long span = std::min(p.rank_len, p.g_end - p.g_begin);  // positions per rank at most
  const long long nchunks = (span + p.chunk - 1) / p.chunk + (p.flat ? 1 : 0);
  const cudaError_t e = launch_pdl(ns_pack_kernel, dim3(static_cast<unsigned>(nchunks), p.S), dim3(PACK_THREADS), 0,
                                  st, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace nsk
