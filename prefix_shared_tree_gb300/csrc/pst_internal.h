// Internal data structures of libpst shared by the host planner and the
// device kernels. Not part of the public ABI (see include/pst.h).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "pst.h"

namespace pst {

// Rows of the tensor-core PAC per thread block: 128 for the mma.sync kernel
// (8 warps x 16 rows), 256 for the tcgen05 kernel (two M=128 halves).
constexpr int kTcRowsPerBlock = 128;
constexpr int kUmmaRowsPerBlock = 256;
inline int tc_rows_per_block(const pst_plan_opts& o) {
    return o.tc_engine == 1 ? kTcRowsPerBlock : (o.tc_block_rows == 128 ? 128 : kUmmaRowsPerBlock);
}
// Rows of the CUDA-core PAC per thread block (largest row tile).
constexpr int kCcRowsPerBlock = 8;
// tcgen05 thin PAC: rows per head of an item (at most; 4 or 8) and kv heads
// per item.
constexpr int kThinRows = 8;
constexpr int kThinHeads = 8;
// KV tokens per pipeline stage of the CUDA-core and mma.sync PAC kernels
// (4 boxes of 16 rows) and of the tcgen05 PAC (8 boxes).
constexpr int kTileTokens = 64;
constexpr int kTcTileTokens = 128;
// Default of pst_plan_opts::p_bf16_min_tokens.
constexpr int kPBf16MinTokens = 1024;
// Rows of one TMA box (page_size must be a multiple).
constexpr int kBoxRows = 16;
// Maximum tokens of a chunk that carries a per-query 64-bit mask.
constexpr int kMaskTokens = 64;

// One KV chunk: a token range of a node, or a packed page-contiguous subtree
// whose visibility is given by one 64-bit mask per query.
struct DevChunk {
    int32_t page_base;  // index into pages[] of the chunk's page list entry 0
    int32_t pos_begin;  // page-space position of chunk token 0 (row in entry 0 + 16*k)
    int32_t n_tok;      // tokens in the chunk
    int32_t q_base;     // index into chunk_q[] of the chunk's first query
    int32_t n_q;        // queries grouped with this chunk
    int32_t part_base;  // partial row of (chunk query 0, q-head 0); row = base + qi*Hq + h
    int32_t mask_base;  // -1: every query sees every token; else index into masks[]
    int32_t r_tile;     // rows per block (per kv head): CUDA-core PAC 1, 2, 4 or 8; thin PAC 4 or 8;
                        // tensor-core 128 or 256
};
static_assert(sizeof(DevChunk) == 32, "DevChunk layout");

// One PAC thread block: a chunk, a kv head and a block of rows.
struct DevItem {
    int32_t chunk;
    int16_t kv_head;
    int16_t row_block;
};
static_assert(sizeof(DevItem) == 8, "DevItem layout");

// Byte offsets of the workspace sections (all 256-aligned).
struct WsLayout {
    int64_t status = 0;      // int32 device status word, then kNumCounters work counters
    int64_t items = 0;
    int64_t chunks = 0;
    int64_t pages = 0;
    int64_t chunk_q = 0;
    int64_t masks = 0;
    int64_t merge_ptr = 0;
    int64_t merge_row = 0;
    int64_t tree_pages = 0;  // int32: every page some node uses, once (the MLA rebuild's work list)
    int64_t meta_end = 0;    // metadata [status, meta_end) is uploaded once
    int64_t part_o = 0;      // fp32 [n_part_rows][d]
    int64_t part_lse = 0;    // fp32 [n_part_rows] (log2 domain)
    int64_t total = 0;
};

// Device-side view of a bound plan, passed by value to the kernels.
struct DevPlan {
    const DevItem* items;
    const DevChunk* chunks;
    const int32_t* pages;
    const int32_t* chunk_q;
    const uint64_t* masks;
    const int32_t* merge_ptr;
    const int32_t* merge_row;
    float* part_o;
    float* part_lse;
    int32_t* status;
    int32_t* counters;  // work-queue counters of the persistent PAC launches (zeroed by POR)
    int32_t n_queries, n_q_heads, n_kv_heads, group, d, page_size;
    float scale_log2;  // log2(e) / sqrt(d)
    int32_t debug_stall;  // test only: see pst_plan_opts::debug_stall
};

// PAC kinds of the cost model: CUDA core, tensor core with P rounded once to
// bf16, tensor core with exact (hi + lo) P, tcgen05 thin PAC.
constexpr int kCostKinds = 4;

// Work-queue counters after the status word (one per persistent launch).
constexpr int kNumCounters = 8;

// Device status word codes (bit flags).
enum : int32_t {
    kStatusWaitTimeout = 1,  // a bounded mbarrier wait gave up
    kStatusBadIndex = 2,     // a page or row index failed its range check
};

struct Tree {
    int32_t n_nodes = 0;
    int32_t page_size = 16;
    int64_t num_pages = 0;
    std::vector<int32_t> len, parent, first_offset, depth, preorder;
    std::vector<int64_t> page_ptr;
    std::vector<int32_t> page_ids;
    std::vector<std::vector<int32_t>> children;
    std::vector<int32_t> unique_pages;   // every page some node uses, once, ascending
};

struct HostChunk {
    int32_t task;          // index into tasks
    int32_t node;          // node id, or -1 for a packed subtree
    int32_t tok_begin;     // token range inside the node (node chunks)
    int32_t tok_end;
    int32_t kind;          // 0 CUDA-core, 1 tensor-core
    DevChunk dev;
};

struct Task {              // CoDec T[i] = (n_q[i], n[i]) per kv head
    int32_t node;          // -1 for a packed subtree
    int32_t group;         // packed group index or -1
    int32_t n_q;           // queries sharing it
    int32_t rows;          // n_q * G
    int32_t n_tok;
    int32_t kind;
    int32_t b_k = 1;       // KV-axis splits
    int32_t max_splits = 1;
};

struct PackedGroup {
    int32_t root;                      // the node whose descendants are packed
    std::vector<int32_t> nodes;        // packed nodes in chunk order
    std::vector<int32_t> tok_node;     // per chunk token: node
    std::vector<int32_t> tok_t;        // per chunk token: token index in node
    std::vector<int32_t> page_list;    // virtual page list
    int32_t pos_begin = 0;
    std::vector<int32_t> queries;      // ascending
    std::vector<uint64_t> mask;        // per query
};

void set_error(const std::string& msg);
int fail(int code, const std::string& msg);

// cost model (plan.cpp)
double cost_estimate(int kind, double rows, double tokens);

}  // namespace pst

struct pst_tree {
    pst::Tree t;
};

struct pst_plan {
    // inputs
    int32_t n_queries = 0, hq = 0, hkv = 0, group = 0, d = 0;
    pst_dtype dtype = PST_BF16;
    int32_t page_size = 16;
    int64_t num_pages = 0;
    int32_t n_nodes = 0;
    pst_plan_opts opts{};
    // index (CSR)
    std::vector<int32_t> qpath_ptr, qpath_node, nodeq_ptr, nodeq;
    // partition
    std::vector<pst::Task> tasks;
    std::vector<pst::PackedGroup> groups;
    std::vector<pst::HostChunk> chunks;
    std::vector<int32_t> pages;        // tree pages + packed virtual page lists
    std::vector<int32_t> chunk_q;
    std::vector<uint64_t> masks;
    std::vector<int32_t> merge_ptr, merge_row;
    std::vector<int32_t> tree_pages;   // ascending ids of the pages the tree's nodes use
    std::vector<pst::DevItem> items;   // tensor-core items first, then CUDA-core
    int64_t n_tc_items = 0, n_cc_items = 0;
    // Tensor-core items come in four launch groups, in this order: P rounded
    // once with more than 128 rows per block (both row halves), P once with at
    // most 128, exact P (nodes shorter than opts.p_bf16_min_tokens) with more
    // than 128, exact P with at most 128. Counts per group.
    int64_t tc_group_cnt[4] = {0, 0, 0, 0};
    // thin-chunk items: with the thin PAC all in class 0 (one launch); with the
    // CUDA-core PAC grouped by row tile 8, 4, 2, 1. Offsets into items[] and counts
    int64_t cc_class_off[4] = {0, 0, 0, 0}, cc_class_cnt[4] = {0, 0, 0, 0};
    bool thin = false;   // thin chunks run on the tcgen05 thin PAC
    int64_t n_part_rows = 0;
    // stats
    double plan_us = 0, makespan_us = 0, cost_l_us = 0;
    int32_t num_slots = 0;
    int64_t kv_tokens_read = 0, unique_tokens = 0;
    // device binding
    pst::WsLayout ws;
    std::vector<uint8_t> meta_blob;    // staged metadata image [0, meta_end)
    void* d_ws = nullptr;
    // side streams and fork/join events (cudaStream_t / cudaEvent_t) that run
    // the PAC launch groups (tensor-core, tensor-core exact-P, CUDA-core) side
    // by side; created on first use
    mutable void* side_stream[4] = {nullptr, nullptr, nullptr, nullptr};
    mutable void* ev_fork = nullptr;
    mutable void* ev_join[4] = {nullptr, nullptr, nullptr, nullptr};
    // cached TMA descriptors (built on first decode for a pool pointer)
    mutable const void* tmap_k_ptr = nullptr;
    mutable const void* tmap_v_ptr = nullptr;
    // per pool: the 3-D map of the tensor-core and CUDA-core PACs, then (bf16,
    // d = 128) the 5-D maps of the thin PAC (8-head boxes) and of the tcgen05
    // PAC's V tiles (4 KB page boxes)
    alignas(64) mutable unsigned char tmap_k[384];
    alignas(64) mutable unsigned char tmap_v[384];
    // Q for the tcgen05 PAC (boxes of 128 rows x 64 channels), when the plan's
    // shape allows one (bf16, a GQA group that divides 128)
    mutable const void* tmap_q_ptr = nullptr;
    alignas(64) mutable unsigned char tmap_q[128];
};
