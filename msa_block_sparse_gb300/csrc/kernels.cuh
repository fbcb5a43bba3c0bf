// Launchers of the compute kernels (one .cu file each) and the workspace
// layouts of the calls that need scratch memory.
#pragma once
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace msa {

// Longest supported sequence: the per-tile block bitmaps hold 1024 blocks.
constexpr int kMaxSeqlen = 1024 * kBlock;

// ---------------------------------------------------------------- prologue
struct PrologueJob {
  const __nv_bfloat16* x;    // [T, H, 128] input
  __nv_bfloat16* y;          // [T, H, 128] output (may equal x)
  const __nv_bfloat16* w;    // [128]
  int H;
};
msa_status_t launch_prologue(const PrologueJob* jobs, int njobs, const int32_t* cu, int S,
                             int T, float rope_base, float eps, cudaStream_t stream);
struct DecodeAppendJob {
  const __nv_bfloat16 *q, *q_idx, *k, *v, *k_idx;        // new token, pre-norm [B, H, 128]
  const __nv_bfloat16 *w_q, *w_qi, *w_k, *w_ki;          // [128]
  __nv_bfloat16 *q_out, *q_idx_out;                       // [B, Hq / Hkv, 128]
  __nv_bfloat16 *k_cache, *v_cache, *kidx_cache;          // [page, Hkv, 128, 128]
  int Hq, Hkv;
};
msa_status_t launch_decode_append(const DecodeAppendJob& j, const int32_t* block_table,
                                  const int32_t* cache_lens, int B, int num_pages,
                                  int max_pages, float rope_base, float eps,
                                  cudaStream_t stream);
size_t prologue_bwd_workspace_floats(int T);
msa_status_t launch_prologue_bwd(const __nv_bfloat16* x, const __nv_bfloat16* dy,
                                 __nv_bfloat16* dx, float* dw, const __nv_bfloat16* w, int H,
                                 const int32_t* cu, int S, int T, float rope_base, float eps,
                                 float* dw_part, cudaStream_t stream);

// ---------------------------------------------------------------- index select
// Work units (query tile, index head, chunk of earlier key blocks): at most
// tiles x Hi + kSelUnitsBeyondTiles of them (the plan sizes the chunks so).
constexpr int kSelUnitsBeyondTiles = 640;
struct SelWorkspace {
  int4* units;         // [max_units] (sequence start, query block, first block, end block)
  int4* aux;           // [max_units] (tile x Hi + head, chunks, first slot, chunk | rows << 16)
  int* num_units;      // [1]
  int* claim;          // [1] next unit to claim
  int* merge_ctr;      // [max_tiles * Hi] chunks of the tile finished
  int* tile_start;     // [S + 1] first tile of each sequence
  unsigned long long* part;   // [max_units][15][128] top-15 lists (entry keys) of split tiles' chunks
  int max_units, max_tiles;
};
SelWorkspace carve_select_workspace(WsCursor& ws, int T, int S, int Hi);
msa_status_t launch_index_select(const void* q_idx, const void* k_idx, const int32_t* cu, int S,
                                 int T, int Hi, int max_seqlen, int n_init,
                                 const SelWorkspace& w, int32_t* sel, cudaStream_t stream);

// ---------------------------------------------------------------- sparse forward
// Per (8-token query tile, KV head): word 0 = number of union blocks, words
// 4.. = entries (block << 8) | (bit i: token i of the tile selected the block).
constexpr int kFwdUnionStride = 132;
struct FwdWorkspace {
  Plan plan;
  int* ulist;          // [max_tiles * 16, Hkv, kFwdUnionStride]
  int* tile_ctr;       // [Hkv] next tile to claim, zeroed by fwd_union_kernel
};
FwdWorkspace carve_fwd_workspace(WsCursor& ws, int T, int S, int Hkv);
// A region to zero while the forward runs (e.g. the backward's fp32
// accumulators): `bytes` (a multiple of 16) from the 16-byte aligned `ptr`,
// written by bulk copies from a zeroed shared-memory buffer, plus `nints`
// ints at `ints`.  Empty: ptr null, nints 0.
struct FwdClear {
  void* ptr = nullptr;
  size_t bytes = 0;
  int* ints = nullptr;
  int nints = 0;
};
msa_status_t launch_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const FwdWorkspace& fw, void* o, float* lse,
                               const FwdClear& clear, cudaStream_t stream);

// ---------------------------------------------------------------- sparse backward
// Work items of the KV-major backward: (sequence, key block, segment of
// candidate query tokens), listed key block ascending.
constexpr int kBwdSegment = 256;    // window of candidate query positions per work item

struct BwdWorkspace {
  int4* items;         // [max_items] (s, b, token_begin, token_end) in sequence positions
  int* num_items;      // [1]
  int max_items;
  int* lists;          // [max_items, Hkv, kBwdSegment] positions that selected the item's block
  int* list_len;       // [max_items, Hkv]
  int* order;          // [Hkv, max_items] claim order of the items
  int* lists_done;     // [Hkv] CTAs of bwd_lists_kernel finished (cleared by the Delta kernel)
  float* lsd;          // [T, Hkv, 2, 16]  -lse log2(e) of the group's 16 rows, then -rowsum(dout * o)
  float* dq_acc;       // [T, Hq, 128] fp32
  float* dk_acc;       // [T, Hkv, 128] fp32
  float* dv_acc;       // [T, Hkv, 128] fp32
  int* item_ctr;       // [Hkv] next item to claim (cleared with the accumulators)
};
BwdWorkspace carve_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv, int max_seqlen);
int device_sm_count();
size_t device_l2_bytes();   // L2 cache size of the current device
// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device): the attribute is kept per device.
msa_status_t ensure_smem_ptr(const void* kernel, size_t bytes, const char* name);
template <typename K>
inline msa_status_t ensure_smem(K kernel, size_t bytes, const char* name) {
  return ensure_smem_ptr(reinterpret_cast<const void*>(kernel), bytes, name);
}
// clear_acc = false: the accumulators were cleared beforehand by
// launch_bwd_clear on this workspace.
msa_status_t launch_sparse_bwd(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const BwdWorkspace& ws, void* dq, void* dk, void* dv,
                               bool clear_acc, cudaStream_t stream);
// Zeroes the workspace's fp32 accumulators and item counters (one memset).
msa_status_t launch_bwd_clear(const BwdWorkspace& ws, int Hkv, cudaStream_t stream);

// ---------------------------------------------------------------- decode
struct DecodeWorkspace {
  float* scores;       // [B, Hkv, max_pages] per-block max logits
  int32_t* sel;        // [B, Hkv, 16] selected blocks (ascending, -1 padded)
  float* part_o;       // [B, Hkv, kDecodeSplits, 16, 128] partial outputs
  float* part_ml;      // [B, Hkv, kDecodeSplits, 16, 2] partial (max, sum)
  int max_pages;
};
constexpr int kDecodeSplits = 4;     // the 16 selected blocks are attended in 4 groups
constexpr int kSplitBlocks = kTopK / kDecodeSplits;   // blocks per group
DecodeWorkspace carve_decode_workspace(WsCursor& ws, int B, int Hq, int Hkv, int max_pages);
msa_status_t launch_decode(const void* q, const void* q_idx, const void* k_cache,
                           const void* v_cache, const void* kidx_cache,
                           const int32_t* block_table, const int32_t* cache_lens, int B, int Hq,
                           int Hkv, int num_pages, int max_pages, float scale, int n_init,
                           void* o, int32_t* sel_out, const DecodeWorkspace& ws,
                           cudaStream_t stream);

// ---------------------------------------------------------------- narrow blocks
// 4-token key blocks, head dim 256, 12 query heads per KV head.
constexpr int kQsaMaxSeqlen = 32768;
constexpr int kQsaMaxWords = kQsaMaxSeqlen / 128;   // bitmap words per (token, KV head)
constexpr int kQsaMaxTopk = 1024;
int qsa_mask_words(int max_seqlen);
struct QsaFwdWorkspace {
  Plan plan;           // 10-token query tiles
  uint32_t* masks;     // [T, Hkv, W] selected-block bitmaps
  int W;
  int* ulist;          // [max_tiles, Hkv, ustride]: count, then key tiles
  int ustride;
  int* tile_ctr;       // [Hkv] next query tile to claim (zeroed by qsa_union_kernel)
};
struct QsaBwdWorkspace {
  QsaFwdWorkspace map;
  float2* lsd;         // [T, Hq] (-lse log2 e, -Delta)
  int4* items;         // [max_items] (s, key tile, window, 0)
  int* num_items;
  int max_items;
  int* klist;          // [max_items, Hkv, 129]: count, then query tiles
  int* order;          // [Hkv, max_items] non-empty items, most query tiles first
  int* num_busy;       // [Hkv] non-empty items
  int* item_ctr;       // [Hkv] next item to claim (zeroed by qsa_order_kernel)
  float* dk_acc;       // [T, Hkv, 256] fp32 (scaled)
  float* dv_acc;       // [T, Hkv, 256] fp32, right after dk_acc
};
QsaFwdWorkspace carve_qsa_fwd_workspace(WsCursor& ws, int T, int S, int Hkv, int max_seqlen);
QsaBwdWorkspace carve_qsa_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv,
                                        int max_seqlen);
msa_status_t launch_qsa_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                            const int32_t* cu, int S, int T, int Hq, int Hkv, int topk,
                            int max_seqlen, float scale, const QsaFwdWorkspace& fw, void* o,
                            float* lse, cudaStream_t stream);
msa_status_t launch_qsa_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, const int32_t* sel,
                            const int32_t* cu, int S, int T, int Hq, int Hkv, int topk,
                            int max_seqlen, float scale, const QsaBwdWorkspace& w, void* dq,
                            void* dk, void* dv, cudaStream_t stream);

}  // namespace msa
