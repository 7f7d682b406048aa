// stream.cu -- kernels of the chunk-ready streaming front end ("[RFC]
// Chunk-ready symmetric-buffer protocol for streaming MegaMoE inputs",
// sections "Fixed-capacity ring", "Independent readiness generations",
// "Memory ordering"), single GPU.
//
// Generation of chunk c: (epoch << 32) | (c + 1); chunk c lives in slot
// c % S; the slot is free for chunk c once consumed_gen holds the generation
// of chunk c - S (or (epoch << 32) | 0 for the first S chunks, written by the
// begin kernel).  Publishers store generations with st.release.gpu after the
// payload; readers load them with ld.acquire.gpu before the payload.  Every
// wait is bounded by %globaltimer and degrades to "no work" plus a status bit.
#include <cuda_bf16.h>

#include <algorithm>

#include "nvfp4.cuh"
#include "nvfp4moe_stream.h"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t chunk_gen(uint64_t epoch, int64_t seq) { return (epoch << 32) | (uint64_t)seq; }

// Waits until every word equals its wanted value, at most limit_ns.
__device__ bool wait_gens(const uint64_t* const* words, const uint64_t* want, int nwords, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    bool all = true;
    for (int i = 0; i < nwords; ++i) all = all && ld_acquire_u64(words[i]) == want[i];
    if (all) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// moe_stream_begin: epoch + 1; every slot free for the first S chunks.
__global__ void stream_begin_kernel(StreamArgs r) {
  __shared__ uint64_t epoch;
  if (threadIdx.x == 0) {
    epoch = r.hdr->epoch + 1;
    r.hdr->epoch = epoch;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < r.S; s += blockDim.x) {
    SlotMeta* m = r.meta + s;
    m->done[0] = m->done[1] = 0;
    m->fail[0] = m->fail[1] = 0;
    m->consumed_gen = chunk_gen(epoch, 0);
  }
  __threadfence();
}

// moe_stream_publish: every CTA waits for the slot to be free, copies its
// share of the parts, and counts itself done; the last CTA to finish writes
// the chunk's base and count and releases the parts' generations (or, if a
// CTA gave up waiting, flags the ring and publishes nothing).
__global__ void __launch_bounds__(256) stream_publish_kernel(PublishArgs a) {
  __shared__ int free_ok;
  const int s = (int)(a.r.chunk % a.r.S);
  SlotMeta* m = a.r.meta + s;
  const int cs = a.parts == MOE_STREAM_LAYOUT ? 1 : 0;   // counter set of this publish
  const uint64_t epoch = ld_acquire_u64(&a.r.hdr->epoch);
  if (threadIdx.x == 0) {
    const uint64_t prev = chunk_gen(epoch, a.r.chunk >= a.r.S ? a.r.chunk + 1 - a.r.S : 0);
    const uint64_t* w[1] = {&m->consumed_gen};
    free_ok = wait_gens(w, &prev, 1, a.r.wait_ns) ? 1 : 0;
  }
  __syncthreads();
  if (free_ok) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nthr = (int64_t)gridDim.x * blockDim.x;
    if (a.parts & MOE_STREAM_LAYOUT) {
      const int64_t n16 = (int64_t)a.n * a.H / 8;   // 16-byte vectors of x
      const uint4* src = reinterpret_cast<const uint4*>(a.x);
      uint4* dst = reinterpret_cast<uint4*>(a.slot_x);
      for (int64_t i = tid; i < n16; i += nthr) dst[i] = __ldg(src + i);
    }
    if (a.parts & MOE_STREAM_ROUTE) {
      const int64_t nk = (int64_t)a.n * a.k, ck = a.C * a.k;
      for (int64_t i = tid; i < ck; i += nthr) {
        a.slot_ids[i] = i < nk ? __ldg(a.ids + i) : a.E;   // rows past n: an id the forward skips
        a.slot_w[i] = i < nk ? __ldg(a.w + i) : (uint16_t)0;
      }
    }
  }
  __threadfence();   // this thread's copies, before its CTA counts itself done
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!free_ok) atomicOr(&m->fail[cs], 1);
    __threadfence();
    if (atomicAdd(&m->done[cs], 1) == (int)gridDim.x - 1) {
      __threadfence();
      const bool fail = atomicOr(&m->fail[cs], 0) != 0;
      m->done[cs] = 0;
      m->fail[cs] = 0;
      if (fail) {
        atomicOr(&a.r.hdr->status, MOE_STREAM_PRODUCER_TIMEOUT);
      } else {
        const uint64_t gen = chunk_gen(epoch, a.r.chunk + 1);
        if (a.parts & MOE_STREAM_ROUTE) {
          m->token_base = a.token_base;
          m->n = a.n;
          st_release_u64(&m->route_gen, gen);
        }
        if (a.parts & MOE_STREAM_LAYOUT) st_release_u64(&m->layout_gen, gen);
      }
    }
  }
}

// Before the chunk's forward: both generations published?  Hands the chunk's
// count and base to the finalize through the workspace header.
__global__ void stream_gate_kernel(StreamArgs r, int64_t C, int32_t* ws_hdr) {
  if (threadIdx.x != 0) return;
  const SlotMeta* m = r.meta + (int)(r.chunk % r.S);
  const uint64_t gen = chunk_gen(ld_acquire_u64(&r.hdr->epoch), r.chunk + 1);
  const uint64_t* w[2] = {&m->route_gen, &m->layout_gen};
  const uint64_t want[2] = {gen, gen};
  if (wait_gens(w, want, 2, r.wait_ns)) {
    const int32_t n = m->n;
    ws_hdr[HDR_STREAM_N] = n < 0 ? 0 : (n > C ? (int32_t)C : n);
    *reinterpret_cast<int64_t*>(ws_hdr + HDR_STREAM_BASE) = m->token_base;
    ws_hdr[HDR_STREAM_OK] = 1;
  } else {
    ws_hdr[HDR_STREAM_N] = 0;
    ws_hdr[HDR_STREAM_OK] = 0;
    set_status(ws_hdr + HDR_STATUS, DEVSTAT_STREAM_WAIT);
  }
}

// After the chunk's finalize: the slot may be reused.
__global__ void stream_release_kernel(StreamArgs r, const int32_t* ws_hdr) {
  if (threadIdx.x != 0 || !ws_hdr[HDR_STREAM_OK]) return;
  SlotMeta* m = r.meta + (int)(r.chunk % r.S);
  st_release_u64(&m->consumed_gen, chunk_gen(ld_acquire_u64(&r.hdr->epoch), r.chunk + 1));
}

// The streamed chunk's BF16 finalize: accumulator rows 0 .. n-1 into output
// rows base .. base + n - 1 (n and base from the header), nothing if the gate
// failed or the rows do not fit the output.
__global__ void __launch_bounds__(256) finalize_rows_kernel(const float* __restrict__ acc, uint16_t* __restrict__ out,
                                                            int64_t out_rows, int H, int32_t* ws_hdr) {
  pdl_wait();
  pdl_launch_dependents();
  if (!ws_hdr[HDR_STREAM_OK]) return;
  const int64_t n = ws_hdr[HDR_STREAM_N];
  const int64_t base = *reinterpret_cast<const int64_t*>(ws_hdr + HDR_STREAM_BASE);
  if (n <= 0) return;
  if (base < 0 || base + n > out_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(ws_hdr + HDR_STATUS, DEVSTAT_STREAM_BOUNDS);
    return;
  }
  const int64_t n8 = n * H / 8;
  const float4* src = reinterpret_cast<const float4*>(acc);
  uint4* dst = reinterpret_cast<uint4*>(out + base * H);
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n8; i += (int64_t)gridDim.x * 256) {
    const float4 a = src[2 * i], b = src[2 * i + 1];
    uint32_t w[4];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_stream_begin(const StreamArgs& r, cudaStream_t st) {
  stream_begin_kernel<<<1, 64, 0, st>>>(r);
  return cudaGetLastError();
}

cudaError_t launch_stream_publish(const PublishArgs& a, int num_sms, cudaStream_t st) {
  const int64_t work = std::max<int64_t>((a.parts & MOE_STREAM_LAYOUT) ? (int64_t)a.n * a.H / 8 : 0,
                                         (a.parts & MOE_STREAM_ROUTE) ? a.C * a.k : 0);
  const int64_t want = (work + 255) / 256;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 2));
  stream_publish_kernel<<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_stream_gate(const StreamArgs& r, int64_t C, int32_t* ws_hdr, cudaStream_t st) {
  stream_gate_kernel<<<1, 32, 0, st>>>(r, C, ws_hdr);
  return cudaGetLastError();
}

cudaError_t launch_stream_release(const StreamArgs& r, const int32_t* ws_hdr, cudaStream_t st) {
  stream_release_kernel<<<1, 32, 0, st>>>(r, ws_hdr);
  return cudaGetLastError();
}

cudaError_t launch_finalize_rows(const float* acc, uint16_t* out, int64_t out_rows, int H, int32_t* ws_hdr,
                                 int64_t C, int num_sms, cudaStream_t st) {
  const int64_t want = (C * H / 8 + 255) / 256;
  const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 4));
  void* args[] = {const_cast<float**>(&acc), &out, &out_rows, &H, &ws_hdr};
  return launch_with_pdl((const void*)finalize_rows_kernel, dim3(blocks), dim3(256), 0, st, args);
}

}  // namespace moe
