/*
 * tok.h -- C ABI of the GB300 exact byte-level BPE tokenizer.
 *
 * The operation is the fresh-session GPU path of "TokTier: exact stateful
 * tokenization for agentic LLM serving" (Section 4, "exact GPU
 * tokenization"): bytes in, token ids out, identical to the serial reference
 * tokenizer.  The tokenizer is the two-stage map F = E* . G of Appendix A.1:
 * G splits the UTF-8 text into fragments with a GPT-style pre-tokenizer
 * regex (Section 4.1 recasts that serial regex as a parallel decomposition
 * into runs of letter / digit / whitespace / other code points), then E
 * encodes every fragment on its own with BPE merges in rank order (Section
 * 4.2).  No normaliser, special tokens, truncation or dropout (the
 * assumptions of Appendix A.1).  Output is an id array only, no byte offsets
 * (Section 4.4).  Section 4.3 packages the whole bytes -> ids chain so that
 * a request needs two host synchronisations.  Here the chain is one memset
 * and three kernel launches with no synchronisation between them, on a
 * workspace that grows to the largest input seen and is then reused; a host
 * request synchronises once when its output buffers are pinned (the device
 * writes ids and status straight into them) and twice otherwise (status,
 * then the id copy).
 *
 * Conventions for every function:
 *   - Return 0 (TOK_OK) or a negative TOK_E* code.  Nothing traps or aborts.
 *   - A handle is not reentrant: calls on one handle must not overlap.
 *   - "host" pointers are ordinary CPU memory (pageable or pinned); "device"
 *     pointers are CUDA global memory of the handle's device.
 *   - The library copies everything tok_load is given; all other buffers are
 *     borrowed for the duration of the call only.
 *   - Outputs are undefined when a call fails; tok_last_error() says why.
 *   - A text (or a packed batch) is at most 2^34 - 2 bytes; longer ones are
 *     refused with TOK_EINVAL.
 */
#ifndef TOK_H
#define TOK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tok_handle tok_handle;

enum {
  TOK_OK = 0,
  TOK_EINVAL = -1,   /* bad argument (null pointer, bad pattern id, ...)      */
  TOK_EUTF8 = -2,    /* input is not well-formed UTF-8 (RFC 3629)             */
  TOK_ENOMEM = -3,   /* a device or pinned host allocation failed             */
  TOK_ECUDA = -4,    /* a CUDA runtime call failed                            */
  TOK_EBUF = -5,     /* the output buffer is too small                        */
  TOK_ETIMEOUT = -6, /* a bounded device-side wait gave up (no hang)          */
  TOK_EMERGES = -7   /* vocabulary / merges failed validation                 */
};

/* Pre-tokenizer patterns.  The pages name the cl100k / o200k / DeepSeek
 * families (Section 4.1) without printing them; these are the GPT-2 pattern,
 * the cl100k-style pattern, an o200k-style pattern of this library's own
 * definition (letter runs split where a lower-case or caseless letter is
 * followed by an upper-case one, contractions suffixes of the word before,
 * a symbol run's tail of CR, LF and '/') and a DeepSeek-style pattern of its
 * own definition (the cl100k-style pattern with the letter runs of the CJK
 * scripts, C = letters of script extensions Han, Hiragana, Katakana or
 * Hangul, apart from other letters and without a prefix):
 *   GPT-2:  's|'t|'re|'ve|'m|'ll|'d| ?\p{L}+| ?\p{N}+| ?[^\s\p{L}\p{N}]+|\s+(?!\S)|\s+
 *   cl100k: (?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\r\n\p{L}\p{N}]?\p{L}+|\p{N}{1,3}
 *           | ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+
 *   o200k:  [^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]*[\p{Ll}\p{Lm}\p{Lo}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*
 *           |[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*
 *           |\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n/]*|\s*[\r\n]+|\s+(?!\S)|\s+
 *   DeepSeek: (?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\r\n\p{L}\p{N}]?(?:(?!C)\p{L})+|(?:(?=C)\p{L})+
 *           |\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+        */
enum { TOK_PAT_GPT2 = 0, TOK_PAT_CL100K_STYLE = 1, TOK_PAT_O200K_STYLE = 2, TOK_PAT_DEEPSEEK_STYLE = 3 };

/* Flag ORed into tok_load's pattern_id: Section 4.2's whole-word lookup
 * (Llama-style `ignore_merges`): a fragment whose bytes are a token of the
 * vocabulary is that token, without the merge loop; every other fragment is
 * encoded by BPE as usual.  Needs every token to be at most 255 bytes. */
enum { TOK_IGNORE_MERGES = 0x100 };

/* tok_load -- build a tokenizer on the current CUDA device.
 *
 * vocab_bytes / vocab_off: token t has bytes vocab_bytes[vocab_off[t] ..
 *   vocab_off[t+1]) (host, n_vocab+1 offsets).  Each of the 256 single bytes
 *   must be exactly one token; no two tokens may have equal bytes; tokens are
 *   at most 32767 bytes; n_vocab < 2^20.
 * merges: host array of n_merges (left_id, right_id) pairs in rank order
 *   (rank = index).  The result of a merge is the token whose bytes are
 *   bytes(left) || bytes(right); it must exist.  No pair may repeat.
 *   (Section 4.2: BPE merges applied lowest rank first.)
 * pattern_id: TOK_PAT_GPT2, TOK_PAT_CL100K_STYLE, TOK_PAT_O200K_STYLE or
 *   TOK_PAT_DEEPSEEK_STYLE, optionally ORed with TOK_IGNORE_MERGES.
 * out: receives the handle; free it with tok_free.
 * Errors: TOK_EINVAL, TOK_EMERGES (validation, message in tok_last_error(NULL)),
 *   TOK_ENOMEM, TOK_ECUDA.
 */
int tok_load(const uint8_t* vocab_bytes, const uint64_t* vocab_off, uint32_t n_vocab,
             const uint32_t* merges, uint32_t n_merges, int pattern_id, tok_handle** out);

/* tok_encode -- encode one text (host in, host out), Section 4.3's request:
 * runs the whole bytes -> ids chain on the handle's stream.  A pinned
 * (page-locked) text is read by the first kernel in place, any other is
 * copied to the device first; when ids is pinned and cap >= len the last
 * kernel writes the ids straight into it, otherwise they are copied back.
 * ids: host array of capacity cap.  cap >= len always suffices (a token has
 *   at least one byte).  *n_ids receives the number of ids.
 * Errors: TOK_EUTF8 (tok_error_offset() = offset of the first malformed
 *   byte sequence), TOK_EBUF (*n_ids = the required capacity), TOK_ECUDA,
 *   TOK_ENOMEM, TOK_ETIMEOUT.  Empty input gives 0 ids.
 */
int tok_encode(tok_handle* h, const uint8_t* text, uint64_t len,
               int32_t* ids, uint64_t cap, uint64_t* n_ids);

/* tok_encode_offsets -- tok_encode that also returns where each token starts.
 * The session state of Sections 3.1 and 3.4 keeps every token's byte
 * offsets; Section 4.4's GPU path returns ids only and sends requests that
 * need offsets to the CPU.  Here the device writes them: a fragment's first
 * token starts at the fragment's first byte, every next one where the
 * previous token's bytes end (token k ends at offsets[k+1], the last at len).
 * offsets: host int64 array of capacity cap, filled like ids.
 * Errors: as tok_encode; TOK_EINVAL if offsets is NULL.
 */
int tok_encode_offsets(tok_handle* h, const uint8_t* text, uint64_t len,
                       int32_t* ids, int64_t* offsets, uint64_t cap, uint64_t* n_ids);

/* tok_repair_append -- the encoding of a session after an append, from the
 * session's previous encoding (Section 3.3: repair instead of a full encode;
 * Section 3.4: a session keeps ids and byte offsets).
 * text: host, len bytes = the old text (old_len bytes) followed by the
 *   appended bytes.  old_ids / old_offsets: host, old_n entries: the ids and
 *   token byte offsets of the old text as tok_encode_offsets returns them.
 * The old text is cut at its last position whose previous code point is a
 * letter or a number and whose own code point has another class (looking
 * back at most 1 MiB; with no such position the whole text is encoded).  A
 * fragment starts there whatever follows, so the old tokens before the cut
 * are kept and only text[cut..len) is encoded (Appendix A.2's splice theorem
 * with a certified cut).  The result equals tok_encode_offsets(text).
 * ids / offsets: host, capacity cap; they may be old_ids / old_offsets
 *   themselves (the kept tokens are then not copied).
 * *n_ids: number of ids; *reencoded (may be NULL): bytes encoded anew.
 * Errors: TOK_EINVAL (including old offsets that do not fit the text),
 *   TOK_EBUF (*n_ids = the required capacity), and those of tok_encode.
 */
int tok_repair_append(tok_handle* h, const uint8_t* text, uint64_t old_len, uint64_t len,
                      const int32_t* old_ids, const int64_t* old_offsets, uint64_t old_n,
                      int32_t* ids, int64_t* offsets, uint64_t cap, uint64_t* n_ids,
                      uint64_t* reencoded);

/* tok_encode_batch -- encode n independent texts in one pass (host in, host
 * out).  Item k is texts[k][0..lens[k]); items never interact: every item
 * starts and ends a fragment exactly as a separate tok_encode call would.
 * ids: host array of capacity cap (cap >= sum(lens) suffices), filled with
 *   the items' ids back to back; item_off: host array of n+1 entries, item k's
 *   ids are ids[item_off[k] .. item_off[k+1]).
 * Errors: as tok_encode; TOK_EUTF8 reports the offset within the
 *   concatenation of all items; on TOK_EBUF item_off[n] = the required
 *   capacity.
 */
int tok_encode_batch(tok_handle* h, const uint8_t* const* texts, const uint64_t* lens, uint32_t n,
                     int32_t* ids, uint64_t cap, uint64_t* item_off);

/* tok_encode_device -- the same chain on device-resident buffers, enqueued on
 * `stream` (a cudaStream_t of the handle's device; NULL = the CUDA default
 * stream) without any host synchronisation.
 * d_text: device, len bytes.  d_ids: device, cap >= len int32 (required).
 * d_status: device int64[4], valid once the chain has finished (read it
 * after synchronising with `stream`):
 *   [0] = TOK_OK or a negative code, [1] = number of ids,
 *   [2] = offset of the first malformed UTF-8 sequence (or -1), [3] = reserved.
 * Returns TOK_EINVAL / TOK_EBUF / TOK_ENOMEM / TOK_ECUDA for launch-time
 * problems; data-dependent errors appear in d_status only.
 */
int tok_encode_device(tok_handle* h, const uint8_t* d_text, uint64_t len,
                      int32_t* d_ids, uint64_t cap, int64_t* d_status, void* stream);

/* tok_encode_offsets_device -- tok_encode_device that also writes every
 * token's byte offset (as tok_encode_offsets) to d_offsets (device, int64,
 * capacity cap; NULL: none, which is tok_encode_device).
 */
int tok_encode_offsets_device(tok_handle* h, const uint8_t* d_text, uint64_t len,
                              int32_t* d_ids, int64_t* d_offsets, uint64_t cap,
                              int64_t* d_status, void* stream);

/* tok_encode_batch_device -- device-resident batch.  d_text holds the items
 * back to back; d_item_start (device, n+1 int64) gives item k's bytes as
 * d_text[d_item_start[k] .. d_item_start[k+1]), with d_item_start[0] == 0
 * and d_item_start[n] == total length.  d_item_off (device, n+1 int64)
 * receives the id offsets of the items; d_status as tok_encode_device.
 * total = d_item_start[n] must be passed as `len` (host value).
 */
int tok_encode_batch_device(tok_handle* h, const uint8_t* d_text, uint64_t len,
                            const int64_t* d_item_start, uint32_t n, int32_t* d_ids, uint64_t cap,
                            int64_t* d_item_off, int64_t* d_status, void* stream);

/* tok_pretokenize -- the pre-tokenizer G alone (Section 4.1): writes the byte
 * offset of every fragment start of text[0..len) (host in, host out) to
 * starts (capacity cap; cap >= len suffices) and the count to *n.
 * Errors: as tok_encode.
 */
int tok_pretokenize(tok_handle* h, const uint8_t* text, uint64_t len,
                    int64_t* starts, uint64_t cap, uint64_t* n);

/* tok_pretokenize_batch -- tok_pretokenize over n independent texts packed
 * back to back (as tok_encode_batch packs them); starts are byte offsets into
 * that concatenation.  Every item starts a fragment. */
int tok_pretokenize_batch(tok_handle* h, const uint8_t* const* texts, const uint64_t* lens, uint32_t n,
                          int64_t* starts, uint64_t cap, uint64_t* n_starts);

/* tok_pretokenize_device_noalloc -- the pre-tokenizer G on device buffers for
 * callers that cannot allocate device memory (code inside another framework's
 * memory pool or arena, code that must not trigger the device-wide
 * synchronisation cudaMalloc/cudaFree can cause, hosts with a fixed memory
 * budget).  TokTier describes no such call: it is an integration entry point of
 * this library, not a step of the method.
 * Needs no handle and allocates nothing: its scratch (the status block the
 * boundary kernel writes) lives in a fixed __device__ array of this library
 * that every GPU loading it holds until exit.  Calls on one device share that
 * array: do not run two at once.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with the device current);
 * make that first call before any stream capture.
 * d_text: device, len bytes.  d_start_bits: device uint32 words, at least
 *   ceil(len / 32) of them; bit p % 32 of word p / 32 is set iff a fragment
 *   starts at byte p (bits at p >= len are 0).
 * d_status: device int64[2]: [0] = TOK_OK or TOK_EUTF8, [1] = offset of the
 *   first malformed UTF-8 sequence or -1.
 * Enqueued on `stream` (NULL = the CUDA default stream) with no host sync.
 * Every call shares the one scratch array: calls that overlap on the GPU (on
 * different streams or devices' shared contexts) race and must be serialised
 * by the caller.  An empty text (len == 0) only writes d_status, also
 * without a host sync.
 * Errors (checked on the host before anything is enqueued): TOK_EINVAL
 *   (NULL pointers, an unknown pattern, or len > 2^34 - 2, the bound of
 *   every entry point), TOK_ECUDA (no device, the symbol lookup or a launch
 *   failed).
 */
int tok_pretokenize_device_noalloc(int pattern_id, const uint8_t* d_text, uint64_t len,
                                   uint32_t* d_start_bits, int64_t* d_status, void* stream);

/* tok_last_error -- message of the last failure on h (or of the last failed
 * tok_load when h is NULL).  The string is owned by the library and valid
 * until the next call on h. */
const char* tok_last_error(tok_handle* h);

/* tok_error_offset -- byte offset of the first malformed UTF-8 sequence seen
 * by the last host-side call on h that returned TOK_EUTF8, else -1. */
int64_t tok_error_offset(tok_handle* h);

/* tok_content_hash -- 64-bit FNV-1a hash over the pattern id, the token bytes
 * and the merges (Section 3.1: tokenizers are registered by content hash). */
uint64_t tok_content_hash(tok_handle* h);

/* tok_stage_times -- per-kernel device times of the most recent call made
 * with timing enabled (tok_set_timing).  Writes up to cap entries of
 * milliseconds to ms and the matching kernel names (static strings) to names;
 * returns the number of entries, or a negative code. */
int tok_set_timing(tok_handle* h, int enable);
int tok_stage_times(tok_handle* h, float* ms, const char** names, int cap);

/* tok_launch_count -- number of kernels this handle has launched so far. */
uint64_t tok_launch_count(tok_handle* h);

/* tok_debug_fail_alloc -- test hook for the out-of-memory paths: the k-th
 * device or pinned host allocation that h makes from now on (k >= 1: the
 * workspace, item and offset buffers that calls grow on demand) fails the way
 * cudaMalloc does when the device is full, without being attempted; k = 0
 * disarms the hook.  The call that meets it returns TOK_ENOMEM, frees what it
 * had allocated, and leaves h usable.  Host-side bookkeeping only.
 * Errors: TOK_EINVAL (h is NULL). */
int tok_debug_fail_alloc(tok_handle* h, uint32_t k);

/* tok_debug_grid_wait -- test hook for the device-side wait limit.  The BPE
 * kernel encodes many long fragments (more than 256 bytes) on a group of its
 * CTAs that wait for one another at grid barriers; each wait gives up after
 * a time limit (4 s by default) and the call then returns TOK_ETIMEOUT with
 * the device context intact.  From now on every such barrier of h waits for
 * `extra` arrivals beyond the CTAs that come (extra = 1: a barrier that never
 * completes), and the limit is wait_ms milliseconds (0: the default).
 * extra = 0, wait_ms = 0 restores normal operation.  Host-side bookkeeping
 * only.  Errors: TOK_EINVAL (h is NULL). */
int tok_debug_grid_wait(tok_handle* h, uint32_t extra, uint32_t wait_ms);

/* tok_free -- release the handle and its device memory.  NULL is ignored. */
void tok_free(tok_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* TOK_H */
