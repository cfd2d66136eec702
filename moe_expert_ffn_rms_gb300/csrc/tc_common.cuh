// Device helpers shared by the tcgen05 grouped-GEMM kernels (gemm_tc.cu,
// gemm_nvfp4.cu): work units, acquire loads, proxy fences, pipeline tails,
// and the host tensor-map encoder.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

using namespace ptx;

struct Unit {
  int job, e, nt, row0, rows;
  int split;  // K split of the unit (split-K launches; else 0)
};

// Unit u of a job: expert e has ceil(cnt/chunk) token chunks, each with nt N
// tiles; s_up[e] is the exclusive prefix of units.  Within an expert the N
// tile varies fastest (mt_fast = false), or the token chunk does (mt_fast =
// true: consecutive units share one weight tile).
MOE_DEV Unit unit_of(int u, const int* s_off, const int* s_up, int E, int nt, int chunk,
                     bool mt_fast = false) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_up[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int local = u - s_up[lo];
  int mt, n;
  if (mt_fast) {
    const int chunks = (s_off[lo + 1] - s_off[lo] + chunk - 1) / chunk;
    n = local / chunks;
    mt = local - n * chunks;
  } else {
    mt = local / nt;
    n = local - mt * nt;
  }
  Unit un;
  un.job = 0;
  un.split = 0;
  un.e = lo;
  un.nt = n;
  un.row0 = s_off[lo] + mt * chunk;
  un.rows = min(chunk, s_off[lo + 1] - un.row0);
  return un;
}

MOE_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MOE_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------ pipeline tails --
// tcgen05.commit arrives on its mbarriers asynchronously.  A CTA must not exit
// while such an arrival is still on its way to its shared memory (the next CTA
// on the SM reuses it), so before teardown each role waits for the arrivals it
// has not consumed yet.

// Producer tail: waits until the MMAs have released the last use of every
// ring slot.  (s, ph) is the producer's position after its last slot; a slot
// never used passes at once.
MOE_DEV bool producer_tail(uint64_t* empty_bar, int stages, int s, uint32_t ph,
                           volatile int* abort) {
  for (int i = 0; i < stages; ++i) {
    if (!mbar_wait(&empty_bar[s], ph ^ 1, abort)) return false;
    if (++s == stages) { s = 0; ph ^= 1; }
  }
  return true;
}

// MMA tail: waits until the epilogues have released every accumulator (nacc
// buffers used round-robin).
MOE_DEV bool accumulator_tail(uint64_t* tempty_bar, int acc, uint32_t aph, volatile int* abort,
                              int nacc = 2) {
  for (int i = 0; i < nacc; ++i) {
    if (!mbar_wait(&tempty_bar[acc], aph ^ 1, abort)) return false;
    if (++acc == nacc) { acc = 0; aph ^= 1; }
  }
  return true;
}

// After an abort: waits, bounded, for the copies of the last arming of every
// slot (bit i of `armed`; its phase parity in bit i of `armed_ph`), whether or
// not the MMAs consumed them.
MOE_DEV void drain_armed(uint64_t* full_bar, int stages, uint32_t armed, uint32_t armed_ph) {
  for (int i = 0; i < stages; ++i) {
    if (!((armed >> i) & 1u)) continue;
    const uint32_t par = (armed_ph >> i) & 1u;
    const long long t0 = clock64();
    while (!mbar_try_wait(&full_bar[i], par) && clock64() - t0 < kSpinLimitCycles) {
    }
  }
}

// Host: 2D tensor map of a row-major [rows, cols] matrix of elem_bytes-wide
// elements, box (box_cols, box_rows), 256-byte L2 promotion, zero OOB fill.
// False if the driver entry point is missing or the encoding is rejected.
bool encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
                int64_t rows, int64_t cols, int box_cols, int box_rows, CUtensorMapSwizzle sw);

}  // namespace tc
}  // namespace moe
