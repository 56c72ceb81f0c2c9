// internal.h -- host/device interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pattn {

// Prefill tiles are BLOCK_M query rows of one head.
constexpr int BLOCK_M = 128;
// Key tile of the prefill kernel.
constexpr int BLOCK_N = 128;

// Header at the start of the workspace (one 256-byte line).
struct WsHeader {
  unsigned status;        // PATTN_DEV_* bits
  int num_prefill_tiles;  // written by the plan kernel
  int prefill_ctas;       // written by the plan kernel: CTAs of the prefill grid
                          // that run (0: all); the decode grid takes the SMs of
                          // the others while prefill runs
  unsigned next_item;     // zeroed by the plan kernel: prefill items claimed past
                          // each CTA's first
  int pad[60];
};

struct Problem {
  const void* q;
  const void* kv;
  const int* block_table;
  const int* seq_lens;
  const int* qsl;
  void* out;
  float scale;
  int H, Hkv, G, D, bs, window, causal, kv_dtype;
  int bs_shift;  // log2(bs) when bs is a power of two, else -1
  float k_scale, v_scale;
  int B, T, mbps, NB, max_q, max_s, splits;
  int bt_stride;     // row stride of block_table (>= mbps; the cascade suffix
                     // pass starts rows past the shared prefix)
  int clear_status;  // the plan kernel clears the status word (else an earlier
                     // kernel of the same call did)
  int long_queries;  // a request may have more queries than keys (the cascade
                     // prefix pass: every token of the batch over the prefix,
                     // not causal); otherwise that is bad metadata
  int decode_rows_only;  // the decode kernel serves the query_len == 1 rows and
                         // leaves every other request's rows untouched and
                         // unreported (they belong to another call)
  // Partial-result mode (cascade passes): when set, rows are written as
  // normalised fp32 o [T][H][D] and lse [T][H] (log2 units) instead of out.
  float* o32;
  float* lse32;
  const float* sinks;  // [H] attention-sink logits (natural-log units) or null; used
                       // only where a final output row is normalised
  int kv_chunks;     // prefill in partial-result mode: each row item's key
                     // tiles are cut into this many contiguous chunks, one CTA
                     // and one (o, lse) partial each ([T][H][kv_chunks])
  // workspace views
  WsHeader* hdr;
  int2* tiles;       // (request, row-item) pairs sorted by cost, descending
  int* decode_order; // [B] requests by decreasing visible decode length (decode
                     // rows first); null: request order
  int max_tiles;     // capacity of tiles[]
  int rows_per_item; // query rows of one prefill work item (128 or 256)
  unsigned* counters;  // [B][Hkv]: partitions of a (request, KV-head group) done
  float* o_part;     // [B][H][splits][D]  (splits > 1)
  float* lse_part;   // [B][H][splits]     (log2 domain)
  cudaStream_t stream;
  // Programmatic dependent launch (host-side choices):
  int pdl_launch;   // the decode kernel may start before the previous kernel in
                    // the stream has finished
  int pdl_wait;     // ...and waits for it (griddepcontrol.wait) before it touches
                    // the status word or the partition counters, which that
                    // kernel clears
  int pdl_trigger;  // the prefill kernel lets its dependent start once all of
                    // its CTAs are running (decode CTAs then take the SMs that
                    // finished prefill CTAs leave)
  // Co-scheduling of a mixed batch (host-side choice and cost model): the
  // plan kernel leaves the prefill kernel only as many CTAs (one per SM) as
  // balance the two kernels, and the decode kernel, a programmatic dependent,
  // runs on the other SMs at the same time.
  int co_schedule;
  int num_sms;
  float pf_us_per_tile;    // prefill: us per key tile of one item, per SM
  float dec_bytes_per_us;  // decode: K/V bytes per us one SM streams (two CTAs)
  float hbm_bytes_per_us;  // decode: HBM bytes per us available beside prefill
#ifdef PATTN_WAIT_TEST
  // Wait-test build only: 1 = CTA 0 of the prefill kernel posts no bytes and
  // issues no copy for the first K tile it streams; 2 = CTA 0 of the decode
  // kernel does the same for its first unit.  The wait for that tile then runs
  // out (a barrier phase that nothing completes), which is how the tests reach
  // the timeout path without faulting or hanging anything.
  int test_skip;
#endif
};

#ifdef PATTN_WAIT_TEST
// Wait-test build only: sets Problem::test_skip for the calls that follow
// (0 turns it off).  Exported as pattn_test_set_wait_skip.
extern "C" void pattn_test_set_wait_skip(int mode);
int test_wait_skip();
#endif

// Workspace layout for a problem (offsets in bytes, 256-byte aligned).
// The header and the counters come first, so one memset of counters_end
// bytes clears both.
struct WsLayout {
  size_t counters_off, counters_end, tiles_off, order_off, o_part_off, lse_off, total;
  int max_tiles;
};
WsLayout workspace_layout(int B, int T, int H, int Hkv, int D, int max_q, int splits);

// Attention over a DiffKV cache ([NB][bs][Hkv][dk + dv], K then V per row):
// p.D is dk; out is [T][H][dv].
cudaError_t launch_diffkv(const Problem& p, int dk, int dv);
// The generic (SIMT) kernel over a DiffKV cache; skip_decode leaves the rows
// of requests with query_len 1 to the tensor-core decode kernel.
cudaError_t launch_generic(const Problem& p, int dk, int dv, bool skip_decode);
// The decode rows of a DiffKV batch on the tensor cores (mma.sync), for head
// sizes that diffkv_decode_supported accepts (multiples of 64).
bool diffkv_decode_supported(int dk, int dv);
cudaError_t launch_diffkv_decode(const Problem& p, int dk, int dv);
// TMA tensor map over a DiffKV cache [NB][bs][Hkv][dk + dv] (16-bit) viewed as
// [NB * bs rows][(dk + dv) / 64 chunks of 64 elements][Hkv]; a box is 16 rows
// x `chunks` chunks of one head, landing chunk-major with the 128-byte swizzle.
bool encode_diffkv_map(CUtensorMap* map, const void* cache, int kv_dtype, int dk, int dv, int Hkv,
                       int bs, int NB, int chunks);

// Kernel launchers; each returns the launch's cudaError_t.
cudaError_t launch_plan(const Problem& p);
// Decode-only calls: clears the status word and the partition counters and
// writes p.decode_order, in a kernel that the decode kernel may follow as a
// programmatic dependent.
cudaError_t launch_decode_prep(const Problem& p);
cudaError_t launch_decode(const Problem& p, const CUtensorMap& kv_map);
cudaError_t launch_prefill(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map);
// The prefill kernel's TMA tensor maps over the KV cache [2 * NB][bs][Hkv][D].
// A 16-bit cache (128-byte swizzle): for the K copies, 4-D {D, KV head, slot,
// block} with a box of box_rows slots of one head and one 64-element d half;
// for the V copies (v_groups), 5-D {64, row of a 16-slot group, d half, KV
// head, group} over the cache's groups (block * bs / 16 + slot / 16), with a
// box of box_rows / 16 groups of one head, both d halves, which lands as
// [group][d half][16 rows][128 bytes].  An e4m3 cache: 4-D {D bytes, KV head,
// slot, block}, one box = box_rows whole rows of one head, unswizzled
// (v_groups unused).  Returns false if the driver entry point is missing or
// rejects the map.
bool encode_kv_map(CUtensorMap* map, const void* kv_cache, int kv_dtype, int D, int Hkv, int bs,
                   int NB, int box_rows, bool v_groups);
// q's map (encode_q_map) and the K and V maps of a prefill launch.
bool encode_prefill_maps(CUtensorMap* qmap, CUtensorMap* kmap, CUtensorMap* vmap, const void* q,
                         const void* kv_cache, int kv_dtype, int H, int D, int T, int Hkv, int bs,
                         int NB);

// TMA tensor map for the decode kernel: one box is 16 rows of a group of
// `heads` KV heads (both d halves for 16-bit data), laid out in shared memory
// as [d half][head][row][128 bytes] (16-bit) or [head][row][row bytes] (e4m3).
bool encode_decode_map(CUtensorMap* map, const void* kv_cache, int kv_dtype, int D, int Hkv,
                       int bs, int NB, int heads);
// KV heads one decode CTA serves (4, 2 or 1: the largest dividing Hkv whose
// 16-key K + V unit fits in 16 KB).
int decode_heads_per_cta(int Hkv, int D, int kv_dtype);

// Cascade attention: the metadata set-up before the two passes, and the
// log-sum-exp merge of their partial results into out.
cudaError_t launch_cascade_setup(WsHeader* hdr, const int* qsl, const int* seq_lens, int B,
                                 int prefix, int* pre_qsl, int* pre_sl, int* suf_sl,
                                 cudaStream_t stream);
cudaError_t launch_cascade_merge(const float* o_a, const float* lse_a, int chunks_a,
                                 const float* o_b, const float* lse_b, void* out, const int* qsl,
                                 int B, int T, int H, int D, bool half, const float* sinks,
                                 cudaStream_t stream);

// Query rows one prefill CTA covers: two heads x 128 rows when the GQA group
// size is even, else one head x 256 rows.
int prefill_rows_per_item(int G);

}  // namespace pattn
