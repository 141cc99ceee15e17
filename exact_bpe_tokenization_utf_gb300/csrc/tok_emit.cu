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

// The end of an encode, one thread: an inconsistency the thread found (a
// bug upstream), recorded for the host path and stored in the caller's status
// at once; and, by the last chunk's thread 0, the number of ids, the offsets
// of the items that start at the text end and the rest of the caller's
// status, written without waiting for the other CTAs: the boundary kernel set
// the status code to OK before any stage ran, and the code only ever changes
// to an error (the earlier kernels' errors are final when this kernel
// starts, this kernel's are stored by the thread that finds them), so a late
// store of the code cannot hide an error.
__device__ __noinline__ void emit_tail(const Call& c, DevStatus* st, bool bug, bool last, unsigned long long n_ids) {
  if (bug) {
    set_error(st, ST_EINTERNAL);
    if (c.user_status) c.user_status[0] = ST_EINTERNAL;
  }
  if (!last) return;
  st->n_ids = n_ids;
  if (c.item_off) {
    for (int k = c.n_items; k >= 0 && c.item[k] >= c.n; --k) c.item_off[k] = (long long)n_ids;
  }
  if (!c.user_status) return;
  const long long eo = err_offset(c.epoch, st->err_off);
  const long long code = eo >= 0 ? (long long)ST_EUTF8 : (long long)st->code;
  if (code != ST_OK) c.user_status[0] = code;
  c.user_status[1] = (long long)n_ids;
  c.user_status[2] = eo;
  c.user_status[3] = 0;
}

}  // namespace

// block-wide exclusive sum of v and the sum of u over the CTA, in one pass
__device__ __forceinline__ int block_excl_sum_and_total(int v, unsigned long long u, int* total_v,
                                                        unsigned long long* total_u, int* sh,
                                                        unsigned long long* sh64) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
  unsigned long long su = u;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
    su += __shfl_xor_sync(0xffffffffu, su, off);
  }
  if (lane == 31) sh[warp] = inc;
  if (lane == 0) sh64[warp] = su;
  __syncthreads();
  int pre = 0, tot = 0;
  unsigned long long tu = 0;
#pragma unroll
  for (int k = 0; k < B_THREADS / 32; ++k) {
    const int x = sh[k];
    pre += k < warp ? x : 0;
    tot += x;
    tu += sh64[k];
  }
  *total_v = tot;
  *total_u = tu;
  __syncthreads();
  return pre + inc - v;
}

// K5: the ids of the fragments that start in one 512-byte chunk.  Thread t
// owns bytes 4t .. 4t + 3 of the chunk and the fragments that start there:
// their id counts are in its registers after the up-front loads, so one scan
// gives every fragment's place.  Fragments of more than 8 ids are copied by
// the whole CTA.
template <bool OFFS, bool STAGED>
__global__ void __launch_bounds__(B_THREADS, OFFS ? 10 : 16) k_emit(Call c, Workspace ws, DevVocab V) {
  constexpr int MAX_BIG = BCHUNK / 8;  // fragments of more than 8 ids have 9 bytes or more
  constexpr int STAGE = 2 * BCHUNK;        // ids of a chunk staged for coalesced stores
  __shared__ __align__(16) int tk[BCHUNK];  // tok of every byte of the chunk
  __shared__ int sid[STAGED ? STAGE : 1];   // the chunk's ids, in order, when they go to host memory and fit
  __shared__ int idb[BCHUNK];               // ids of the chunk before each fragment start (batch item offsets)
  __shared__ int big_a[MAX_BIG], big_k[MAX_BIG], big_o[MAX_BIG];
  __shared__ int scan[B_THREADS / 32];
  __shared__ unsigned long long scan64[B_THREADS / 32];
  __shared__ int s_item, s_nbig;
  const int tid = threadIdx.x, T = B_THREADS;
  // a programmatic dependent of the engine kernel: wait for its writes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long nch = n_bchunks(c.n);
  DevStatus* st = ws.st;
  const long long chunk = blockIdx.x;
  const long long r0 = chunk * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  if (tid == 0) s_nbig = 0;
  // every load this CTA needs, issued together: the counts and ids of the
  // thread's bytes (positions past the text end, or that start no fragment,
  // are read but not used; the workspace holds whole chunks), its bits of
  // the bitmask, and the totals before the chunk (group totals before its
  // group, chunk totals before it in its group)
  static_assert(BCHUNK == 4 * B_THREADS, "one int4 of counts and ids per thread");
  const int4 cnt4 = reinterpret_cast<const int4*>(ws.fcnt + r0)[tid];
  const int4 tk4 = reinterpret_cast<const int4*>(ws.tok + r0)[tid];
  const int q0 = 4 * tid;
  uint32_t mine = 0;
  if (r0 + q0 < r1) {
    mine = (ws.pstart[(r0 >> 5) + (q0 >> 5)] >> (q0 & 31)) & 0xFu;
    if (r1 - (r0 + q0) < 4) mine &= (1u << (r1 - (r0 + q0))) - 1u;
  }
  unsigned long long part = 0;
  const long long grp = chunk / CTOT_GROUP;
  for (long long i = tid; i < grp; i += T) part += ws.gtot[i];
  for (long long i = grp * CTOT_GROUP + tid; i < chunk; i += T) part += ws.ctot[i];
  const uint32_t my_total = ws.ctot[chunk];
  reinterpret_cast<int4*>(tk)[tid] = tk4;
  // id counts of the thread's fragments: between 1 and (bytes to the text
  // end); anything else would be a bug upstream, reported instead of
  // written out of bounds
  int cn[4] = {cnt4.x, cnt4.y, cnt4.z, cnt4.w};
  bool bug = false;
  int ids = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!((mine >> q) & 1u)) { cn[q] = 0; continue; }
    if (cn[q] < 1 || cn[q] > c.n - (r0 + q0 + q)) {
      bug = true;
      cn[q] = 0;
    }
    ids += cn[q];
  }
  int total = 0;
  unsigned long long base = 0;  // ids before this chunk
  int o = block_excl_sum_and_total(ids, part, &total, &base, scan, scan64);
  if ((uint32_t)total != my_total) {  // the counts disagree with the chunk total: a bug upstream
    bug |= tid == 0;
    total = 0;
  }
  // ids in text order: fragments of up to 8 ids by their thread, longer ones
  // by the CTA.  When the output is host memory, a chunk's ids that fit in
  // shared memory are staged there and stored in one coalesced pass (the
  // scattered stores of the threads cost far more over the host link)
  const bool staged = STAGED && total <= STAGE;
  if (total > 0) {
#pragma unroll(OFFS ? 1 : 4)
    for (int q = 0; q < 4; ++q) {
      if (!((mine >> q) & 1u)) continue;
      const int k = q == 0 ? cn[0] : q == 1 ? cn[1] : q == 2 ? cn[2] : cn[3];
      const int a0 = q0 + q;
      const long long a = r0 + a0;
      if (c.item_off) idb[a0] = o;
      if (k <= 8) {
        // ids from the staged copy while they lie in the chunk
        for (int j = 0; j < k; ++j) {
          const int id = a0 + j < BCHUNK ? tk[a0 + j] : ws.tok[a + j];
          if (staged) sid[o + j] = id;
          else c.out[base + o + j] = id;
        }
        if (OFFS) {
          long long off = a;
          for (int j = 0; j < k; ++j) {
            c.out_off[base + o + j] = off;
            off += __ldg(V.tok_len + (a0 + j < BCHUNK ? tk[a0 + j] : ws.tok[a + j]));
          }
        }
      } else if (k > 0) {
        const int bi = atomicAdd(&s_nbig, 1);
        if (bi < MAX_BIG) {
          big_a[bi] = a0;
          big_k[bi] = k;
          big_o[bi] = o;
        } else {
          bug = true;
        }
      }
      o += k;
    }
  }
  __syncthreads();
  const int nbig = min(s_nbig, MAX_BIG);
  for (int b = 0; b < nbig; ++b) {
    const long long a = r0 + big_a[b];
    const int k = big_k[b];
    const unsigned long long ob = base + (unsigned long long)big_o[b];
    for (int j = tid; j < k; j += T) {
      if (staged) sid[big_o[b] + j] = ws.tok[a + j];
      else c.out[ob + j] = ws.tok[a + j];
    }
    if (OFFS) {
      // offsets: exclusive scan of the token lengths, one tile of T ids at a time
      long long carry = a;
      for (int j0 = 0; j0 < k; j0 += T) {
        const int j = j0 + tid;
        const int len = j < k ? (int)__ldg(V.tok_len + ws.tok[a + j]) : 0;
        int tile = 0;
        const int ex = block_excl_sum_t(len, &tile, scan);
        if (j < k) c.out_off[ob + j] = carry + ex;
        carry += tile;
      }
    }
  }
  if (staged && total > 0) {
    __syncthreads();
    for (int i = tid; i < total; i += T) c.out[base + i] = sid[i];
  }
  // batch: ids before each item start in this chunk (every item start is a
  // fragment start)
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
      c.item_off[k] = (long long)base + (total > 0 ? idb[x - r0] : 0);
    }
  }
  // the CTA of the last chunk knows the number of ids (the ids before it and
  // its own) and completes the status (emit_tail)
  const bool last = chunk == nch - 1 && tid == 0;
  if (bug || last) emit_tail(c, st, bug, last, base + (unsigned long long)total);
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
  const unsigned g = (unsigned)n_bchunks(c.n);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g);
  cfg.blockDim = dim3(B_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (c.out_off) {
    if (c.out_host) cudaLaunchKernelEx(&cfg, k_emit<true, true>, c, w, v);
    else cudaLaunchKernelEx(&cfg, k_emit<true, false>, c, w, v);
  } else {
    if (c.out_host) cudaLaunchKernelEx(&cfg, k_emit<false, true>, c, w, v);
    else cudaLaunchKernelEx(&cfg, k_emit<false, false>, c, w, v);
  }
}

void launch_status_only(const Call& c, const Workspace& w, cudaStream_t s) {
  k_status_only<<<1, 1, 0, s>>>(c, w);
}

}  // namespace tokgb
