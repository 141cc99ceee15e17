// ID scatter: the ids of all fragments, in text order, as one array ("TokTier:
// exact stateful tokenization for agentic LLM serving", Section 4.3 returns
// an id array; Section 4.4: ids only, no byte offsets).
//
// Each CTA owns a 4 KiB range of bytes and emits the tokens whose first byte
// lies in it.  The number of tokens before the range comes from a
// decoupled look-back over the CTAs' published counts (Merrill and Garland,
// "Single-pass parallel prefix scan with decoupled look-back", 2016): ranges
// are taken in ticket order, so a CTA only waits on CTAs that already run;
// every wait is bounded and reports TOK_ETIMEOUT instead of hanging.
#include "tok_common.cuh"

namespace tokgb {

// look-back word: epoch (30 bits) | flag (2 bits) | value (32 bits)
constexpr unsigned long long LB_AGG = 1ull, LB_INC = 2ull;
constexpr int LB_SPIN_LIMIT = 1 << 22;

__device__ __forceinline__ unsigned long long lb_pack(uint32_t epoch, unsigned long long flag, uint32_t v) {
  return ((unsigned long long)(epoch & 0x3FFFFFFFu) << 34) | (flag << 32) | v;
}

__device__ void write_user_status(const Call& c, const DevStatus* st) {
  if (!c.user_status) return;
  const unsigned long long eo = st->err_off;
  long long code = st->code;
  if (eo != ~0ull) code = ST_EUTF8;
  c.user_status[0] = code;
  c.user_status[1] = (long long)st->n_ids;
  c.user_status[2] = eo == ~0ull ? -1 : (long long)eo;
  c.user_status[3] = 0;
}

__global__ void __launch_bounds__(CHUNK_THREADS) k_emit(Call c, Workspace ws) {
  __shared__ uint32_t s_chunk;
  __shared__ int wsum[CHUNK_THREADS / 32];
  __shared__ unsigned long long s_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long nch = n_chunks(c.n);
  DevStatus* st = ws.st;
  if (tid == 0) s_chunk = atomicAdd(&st->emit_ticket, 1u);
  __syncthreads();
  const long long chunk = s_chunk;
  const long long c0 = chunk * CHUNK;
  const long long p0 = c0 + tid * 16;
  // this thread's 16 token-start flags
  uint32_t mask = 0;
  if (p0 + 16 <= c.n && ((reinterpret_cast<uintptr_t>(ws.tstart) & 15u) == 0)) {
    const uint4 v = *reinterpret_cast<const uint4*>(ws.tstart + p0);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 16; ++q) mask |= ((wv[q >> 2] >> ((q & 3) * 8)) & 1u) << q;
  } else {
    for (int q = 0; q < 16; ++q)
      if (p0 + q < c.n && ws.tstart[p0 + q]) mask |= 1u << q;
  }
  const int cnt = __popc(mask);
  int inc = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int wpre = 0, total = 0;
  for (int k = 0; k < CHUNK_THREADS / 32; ++k) {
    if (k < warp) wpre += wsum[k];
    total += wsum[k];
  }
  const int excl = wpre + inc - cnt;
  if (tid == 0) {
    volatile unsigned long long* lb = ws.lb;
    if (chunk > 0) {
      __threadfence();
      lb[chunk] = lb_pack(c.epoch, LB_AGG, (uint32_t)total);
    }
    unsigned long long prefix = 0;
    bool timed_out = false;
    for (long long j = chunk - 1; j >= 0; --j) {
      unsigned long long v = lb[j];
      int spins = 0;
      while ((uint32_t)(v >> 34) != (c.epoch & 0x3FFFFFFFu)) {
        if (++spins > LB_SPIN_LIMIT) { timed_out = true; break; }
        __nanosleep(64);
        v = lb[j];
      }
      if (timed_out) break;
      prefix += (uint32_t)v;
      if (((v >> 32) & 3ull) == LB_INC) break;
    }
    if (timed_out) atomicExch(&st->code, ST_ETIMEOUT);
    __threadfence();
    lb[chunk] = lb_pack(c.epoch, LB_INC, (uint32_t)(prefix + total));
    s_prefix = prefix;
    if (chunk == nch - 1) st->n_ids = prefix + total;
  }
  __syncthreads();
  const unsigned long long base = s_prefix + excl;
  // ids
  unsigned long long o = base;
  for (int q = 0; q < 16; ++q)
    if ((mask >> q) & 1u) c.out[o++] = ws.sid[p0 + q];
  // item offsets (batch): ids before each item start in this range
  if (c.item_off) {
    __shared__ int s_first;
    if (tid == 0) {
      int lo = 0, hi = c.n_items + 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (c.item[mid] < c0) lo = mid + 1; else hi = mid;
      }
      s_first = lo;
    }
    __syncthreads();
    for (int k = s_first + tid; k <= c.n_items; k += CHUNK_THREADS) {
      const long long x = c.item[k];
      if (x >= c0 + CHUNK || x >= c.n) break;
      // ids before x in this range = token-start flags in bytes [c0, x)
      long long cntb = 0;
      for (long long y = c0; y < x; ++y) cntb += ws.tstart[y] != 0;
      c.item_off[k] = (long long)s_prefix + cntb;
    }
  }
  // the last CTA to finish completes the status
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(&st->emit_done, 1u);
    if (done == (uint32_t)(nch - 1)) {
      __threadfence();
      const unsigned long long nid = *(volatile unsigned long long*)&st->n_ids;
      if (c.item_off) {
        for (int k = c.n_items; k >= 0 && c.item[k] >= c.n; --k) c.item_off[k] = (long long)nid;
      }
      write_user_status(c, st);
    }
  }
}

// empty input: reset the status and report zero ids
__global__ void k_status_only(Call c, Workspace ws) {
  DevStatus* st = ws.st;
  st->code = ST_OK;
  st->err_off = ~0ull;
  st->n_ids = 0;
  if (c.item_off)
    for (int k = 0; k <= c.n_items; ++k) c.item_off[k] = 0;
  write_user_status(c, st);
}

void launch_emit(const Call& c, const Workspace& w, cudaStream_t s) {
  k_emit<<<(unsigned)n_chunks(c.n), CHUNK_THREADS, 0, s>>>(c, w);
}

void launch_status_only(const Call& c, const Workspace& w, cudaStream_t s) {
  k_status_only<<<1, 1, 0, s>>>(c, w);
}

}  // namespace tokgb
