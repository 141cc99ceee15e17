// ID scatter: the ids of all fragments, in text order, as one array ("TokTier:
// exact stateful tokenization for agentic LLM serving", Section 4.3 returns
// an id array; Section 4.4: ids only, no byte offsets).
//
// Every BPE stage left a fragment's ids and their count at the fragment's byte
// offset, and added the count to the total of the 512-byte chunk the fragment
// starts in and to that of the chunk's group of CTOT_GROUP chunks.  K5 takes,
// one CTA per chunk, the ids before the chunk as the sum of the group totals
// before its group and the chunk totals before it in its group, and copies
// the ids of the fragments that start in it, without waiting on another CTA.  On request it also writes every token's
// byte offset: a fragment's first token starts at the fragment, each next
// one where the previous token's bytes end (the session state of Sections
// 3.1 and 3.4 keeps these offsets).
#include "tok_common.cuh"

namespace tokgb {

namespace {

// block-wide exclusive sums (blockDim.x a multiple of 32; sh holds blockDim/32 words)
template <class T>
__device__ __forceinline__ T block_excl_sum_t(T v, T* total, T* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  T pre = 0, tot = 0;
  for (int k = 0; k < nw; ++k) {
    const T x = sh[k];
    pre += k < warp ? x : T(0);
    tot += x;
  }
  *total = tot;
  __syncthreads();
  return pre + inc - v;
}

__device__ void write_user_status(const Call& c, const DevStatus* st) {
  if (!c.user_status) return;
  const long long eo = err_offset(c.epoch, st->err_off);
  long long code = st->code;
  if (eo >= 0) code = ST_EUTF8;
  c.user_status[0] = code;
  c.user_status[1] = (long long)st->n_ids;
  c.user_status[2] = eo;
  c.user_status[3] = 0;
}

}  // namespace

// K5: the ids of the fragments that start in one 512-byte chunk
template <bool OFFS>
__global__ void __launch_bounds__(B_THREADS, 16) k_emit(Call c, Workspace ws, DevVocab V) {
  __shared__ uint32_t bits[BCHUNK / 32];
  __shared__ uint16_t fstart[BCHUNK];
  __shared__ int fcount[BCHUNK];
  __shared__ int foff[BCHUNK];
  __shared__ uint16_t big[BCHUNK];
  __shared__ __align__(16) int cnt[BCHUNK];  // fcnt of every byte of the chunk (meaningful at fragment starts)
  __shared__ __align__(16) int tk[BCHUNK];   // tok of every byte of the chunk
  __shared__ int scan[B_THREADS / 32];
  __shared__ unsigned long long scan64[B_THREADS / 32];
  __shared__ int s_item, s_nbig, s_last;
  const int tid = threadIdx.x, T = B_THREADS;
  const long long nch = n_bchunks(c.n);
  DevStatus* st = ws.st;
  const long long chunk = blockIdx.x;
  const long long r0 = chunk * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  if (tid == 0) s_nbig = 0;
  // every load this CTA needs, issued together: the bitmask, the counts and
  // ids of all the chunk's bytes (positions past the text end, or that start
  // no fragment, are read but not used; the workspace holds whole chunks),
  // and the totals before the chunk (group totals before its group, chunk
  // totals before it in its group)
  static_assert(BCHUNK == 4 * B_THREADS, "one int4 of counts and ids per thread");
  const int4 cnt4 = reinterpret_cast<const int4*>(ws.fcnt + r0)[tid];
  const int4 tk4 = reinterpret_cast<const int4*>(ws.tok + r0)[tid];
  unsigned long long part = 0;
  const long long grp = chunk / CTOT_GROUP;
  for (long long i = tid; i < grp; i += T) part += ws.gtot[i];
  for (long long i = grp * CTOT_GROUP + tid; i < chunk; i += T) part += ws.ctot[i];
  const uint32_t my_total = ws.ctot[chunk];
  if (tid < BCHUNK / 32) {
    const long long p = r0 + 32ll * tid;
    uint32_t v = 0;
    if (p < r1) {
      v = ws.pstart[(r0 >> 5) + tid];
      if (r1 - p < 32) v &= (1u << (r1 - p)) - 1u;
    }
    bits[tid] = v;
  }
  reinterpret_cast<int4*>(cnt)[tid] = cnt4;
  reinterpret_cast<int4*>(tk)[tid] = tk4;
  __syncthreads();
  // the fragments that start in this chunk, and their id counts
  const int q0 = tid * 4;
  const uint32_t mine = (bits[q0 >> 5] >> (q0 & 31)) & 0xFu;
  int nf = 0;
  int idx = block_excl_sum_t(__popc(mine), &nf, scan);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if ((mine >> q) & 1u) fstart[idx++] = (uint16_t)(q0 + q);
  __syncthreads();
  const int FB = (nf + T - 1) / T;
  const int flo = min(tid * FB, nf), fhi = min(flo + FB, nf);
  int ids = 0;
  for (int f = flo; f < fhi; ++f) {
    // a fragment has between 1 and (bytes to the text end) ids; anything else
    // would be a bug upstream, reported instead of written out of bounds
    int k = cnt[fstart[f]];
    if (k < 1 || k > c.n - (r0 + fstart[f])) {
      atomicExch(&st->code, ST_EINTERNAL);
      k = 0;
    }
    fcount[f] = k;
    ids += k;
  }
  int total = 0;
  int o = block_excl_sum_t(ids, &total, scan);
  for (int f = flo; f < fhi; ++f) {
    foff[f] = o;
    o += fcount[f];
  }
  // ids before this chunk
  unsigned long long base = 0;
  block_excl_sum_t(part, &base, scan64);
  if ((uint32_t)total != my_total) {  // the counts disagree with the chunk total: a bug upstream
    if (tid == 0) atomicExch(&st->code, ST_EINTERNAL);
    total = 0;
  }
  __syncthreads();
  // ids in text order: short fragments by their thread, long ones by the CTA
  if (total > 0) {
    for (int f = flo; f < fhi; ++f) {
      const int k = fcount[f];
      const long long a = r0 + fstart[f];
      if (k <= 8) {
        // ids from the staged copy while they lie in the chunk
        const int a0 = fstart[f];
        for (int j = 0; j < k; ++j) c.out[base + foff[f] + j] = a0 + j < BCHUNK ? tk[a0 + j] : ws.tok[a + j];
        if (OFFS) {
          long long off = a;
          for (int j = 0; j < k; ++j) {
            c.out_off[base + foff[f] + j] = off;
            off += __ldg(V.tok_len + (a0 + j < BCHUNK ? tk[a0 + j] : ws.tok[a + j]));
          }
        }
      } else {
        big[atomicAdd(&s_nbig, 1)] = (uint16_t)f;
      }
    }
  }
  __syncthreads();
  for (int b = 0; b < s_nbig; ++b) {
    const int f = big[b];
    const long long a = r0 + fstart[f];
    for (int j = tid; j < fcount[f]; j += T) c.out[base + foff[f] + j] = ws.tok[a + j];
    if (OFFS) {
      // offsets: exclusive scan of the token lengths, one tile of T ids at a time
      long long carry = a;
      for (int j0 = 0; j0 < fcount[f]; j0 += T) {
        const int j = j0 + tid;
        const int len = j < fcount[f] ? (int)__ldg(V.tok_len + ws.tok[a + j]) : 0;
        int tile = 0;
        const int ex = block_excl_sum_t(len, &tile, scan);
        if (j < fcount[f]) c.out_off[base + foff[f] + j] = carry + ex;
        carry += tile;
      }
    }
  }
  // batch: ids before each item start in this chunk
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
    for (int k = s_item + tid; k <= c.n_items; k += T) {
      const long long x = c.item[k];
      if (x >= r1) break;
      int a = 0, b = nf;  // the fragment that starts at x
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (r0 + fstart[mid] < x) a = mid + 1; else b = mid;
      }
      c.item_off[k] = (long long)base + (a < nf ? foff[a] : total);
    }
  }
  // the last CTA to finish completes the status: the number of ids is the
  // sum of the group totals
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&st->emit_done, 1u) == (uint32_t)(nch - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    unsigned long long all = 0;
    for (long long i = tid; i <= (nch - 1) / CTOT_GROUP; i += T) all += ws.gtot[i];
    unsigned long long n_ids = 0;
    block_excl_sum_t(all, &n_ids, scan64);
    if (tid == 0) {
      st->n_ids = n_ids;
      if (c.item_off) {
        for (int k = c.n_items; k >= 0 && c.item[k] >= c.n; --k) c.item_off[k] = (long long)n_ids;
      }
      write_user_status(c, st);
    }
  }
}

// empty input: reset the status and report zero ids
__global__ void k_status_only(Call c, Workspace ws) {
  DevStatus* st = ws.st;
  st->code = ST_OK;
  st->n_ids = 0;
  if (c.item_off)
    for (int k = 0; k <= c.n_items; ++k) c.item_off[k] = 0;
  write_user_status(c, st);
}

void launch_emit(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s) {
  if (c.out_off) k_emit<true><<<(unsigned)n_bchunks(c.n), B_THREADS, 0, s>>>(c, w, v);
  else k_emit<false><<<(unsigned)n_bchunks(c.n), B_THREADS, 0, s>>>(c, w, v);
}

void launch_status_only(const Call& c, const Workspace& w, cudaStream_t s) {
  k_status_only<<<1, 1, 0, s>>>(c, w);
}

}  // namespace tokgb
