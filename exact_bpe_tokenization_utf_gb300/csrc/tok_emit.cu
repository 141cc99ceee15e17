// ID scatter: the ids of all fragments, in text order, as one array ("TokTier:
// exact stateful tokenization for agentic LLM serving", Section 4.3 returns
// an id array; Section 4.4: ids only, no byte offsets).
//
// Each CTA owns a 512-byte chunk and emits the ids of the fragments that start
// in it (K3 left them compacted; a long last fragment's ids come from K4).  The number of tokens before the range comes from a
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

__global__ void __launch_bounds__(B_THREADS) k_emit(Call c, Workspace ws) {
  __shared__ uint32_t s_chunk;
  __shared__ unsigned long long s_prefix;
  __shared__ int s_item;
  const int tid = threadIdx.x;
  const long long nch = n_bchunks(c.n);
  DevStatus* st = ws.st;
  if (tid == 0) s_chunk = atomicAdd(&st->emit_ticket, 1u);
  __syncthreads();
  const long long chunk = s_chunk;
  const long long r0 = chunk * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  const long long first = ws.cm_first[chunk];
  const int n_short = first >= 0 ? ws.cm_count[chunk] : 0;
  const long long lf = first >= 0 ? ws.cm_long[chunk] : -1;
  const int n_long = lf >= 0 ? ws.cm_long_count[chunk] : 0;
  const uint32_t total = (uint32_t)(n_short + n_long);
  if (tid < 32) {
    // warp 0: publish this chunk's count, then look back 32 predecessors at a
    // time until one has published its inclusive prefix
    const int lane = tid;
    volatile unsigned long long* lb = ws.lb;
    const uint32_t ep = c.epoch & 0x3FFFFFFFu;
    if (lane == 0 && chunk > 0) {
      __threadfence();
      lb[chunk] = lb_pack(c.epoch, LB_AGG, total);
    }
    unsigned long long prefix = 0;
    bool timed_out = false;
    for (long long top = chunk - 1; top >= 0; top -= 32) {
      const long long j = top - lane;
      unsigned long long v = j >= 0 ? lb[j] : lb_pack(c.epoch, LB_INC, 0u);
      int spins = 0;
      while (true) {
        const bool ready = (uint32_t)(v >> 34) == ep;
        if (__all_sync(0xffffffffu, ready)) break;
        if (++spins > LB_SPIN_LIMIT) { timed_out = true; break; }
        __nanosleep(64);
        if (!ready) v = lb[j];
      }
      if (timed_out) break;
      const uint32_t inc = __ballot_sync(0xffffffffu, ((v >> 32) & 3ull) == LB_INC);
      const int stop = inc ? __ffs(inc) - 1 : 31;  // nearest predecessor with an inclusive prefix
      unsigned long long x = lane <= stop ? (uint32_t)v : 0ull;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      prefix += x;
      if (inc) break;
    }
    if (lane == 0) {
      if (timed_out) atomicExch(&st->code, ST_ETIMEOUT);
      __threadfence();
      lb[chunk] = lb_pack(c.epoch, LB_INC, (uint32_t)(prefix + total));
      s_prefix = prefix;
      if (chunk == nch - 1) st->n_ids = prefix + total;
    }
  }
  __syncthreads();
  const unsigned long long base = s_prefix;
  // ids: the chunk's fragments, then its long fragment (always its last one)
  for (int j = tid; j < n_short; j += B_THREADS) c.out[base + j] = ws.tok[first + j];
  for (int j = tid; j < n_long; j += B_THREADS) c.out[base + n_short + j] = ws.tok[lf + j];
  // batch: K3 stored the ids before each item start relative to its chunk
  if (c.item_off) {
    if (tid == 0) {
      int a = 0, b = c.n_items + 1;
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (c.item[mid] < r0) a = mid + 1; else b = mid;
      }
      s_item = a;
    }
    __syncthreads();
    for (int k = s_item + tid; k <= c.n_items; k += B_THREADS) {
      if (c.item[k] >= r1) break;
      c.item_off[k] += (long long)base;
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
  k_emit<<<(unsigned)n_bchunks(c.n), B_THREADS, 0, s>>>(c, w);
}

void launch_status_only(const Call& c, const Workspace& w, cudaStream_t s) {
  k_status_only<<<1, 1, 0, s>>>(c, w);
}

}  // namespace tokgb
