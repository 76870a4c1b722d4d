// pst_tree_build: validation and indexing of the KV forest.
//
// CoDec, "KV cache management": the KV cache is a forest of nodes joined by a
// virtual root; an edge p -> c says that p is a prefix of c. Node tokens live in
// fixed-size pages listed per node (PagedAttention block tables, as in the
// shared-prefix techniques blog, section 4.3).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "pst_internal.h"

namespace pst {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

int fail(int code, const std::string& msg) {
    set_error(msg);
    return code;
}

}  // namespace pst

extern "C" const char* pst_last_error(void) { return pst::g_last_error.c_str(); }

extern "C" int pst_tree_build(int32_t n_nodes, const int32_t* node_len, const int32_t* parent,
                              const int64_t* page_ptr, const int32_t* page_ids,
                              const int32_t* first_offset, int32_t page_size, int64_t num_pages,
                              pst_tree** out) {
    using namespace pst;
    if (!out) return fail(PST_EINVAL, "tree_build: out is null");
    *out = nullptr;
    if (n_nodes < 1) return fail(PST_EINVAL, "tree_build: n_nodes must be >= 1");
    if (!node_len || !parent || !page_ptr) return fail(PST_EINVAL, "tree_build: null array");
    if (page_size != 16 && page_size != 32)
        return fail(PST_EUNSUPPORTED, "tree_build: page_size must be 16 or 32");
    if (num_pages < 0 || num_pages > INT32_MAX)
        return fail(PST_ERANGE, "tree_build: num_pages out of range");
    if (page_ptr[0] != 0) return fail(PST_EINVAL, "tree_build: page_ptr[0] must be 0");
    for (int32_t n = 0; n < n_nodes; ++n) {
        if (page_ptr[n + 1] < page_ptr[n])
            return fail(PST_EINVAL, "tree_build: page_ptr must be non-decreasing");
    }
    const int64_t n_page_entries = page_ptr[n_nodes];
    if (n_page_entries > 0 && !page_ids) return fail(PST_EINVAL, "tree_build: page_ids is null");
    if (n_page_entries > INT32_MAX) return fail(PST_ERANGE, "tree_build: too many page entries");

    pst_tree* t = new (std::nothrow) pst_tree();
    if (!t) return fail(PST_ENOMEM, "tree_build: out of memory");
    Tree& T = t->t;
    T.n_nodes = n_nodes;
    T.page_size = page_size;
    T.num_pages = num_pages;
    T.len.assign(node_len, node_len + n_nodes);
    T.parent.assign(parent, parent + n_nodes);
    T.first_offset.assign(n_nodes, 0);
    if (first_offset) T.first_offset.assign(first_offset, first_offset + n_nodes);
    T.page_ptr.assign(page_ptr, page_ptr + n_nodes + 1);
    if (n_page_entries > 0) T.page_ids.assign(page_ids, page_ids + n_page_entries);

    auto bad = [&](int code, const std::string& m) {
        delete t;
        return fail(code, m);
    };
    for (int64_t i = 0; i < n_page_entries; ++i) {
        if (T.page_ids[i] < 0 || T.page_ids[i] >= num_pages)
            return bad(PST_ERANGE, "tree_build: page id " + std::to_string(T.page_ids[i]) +
                                       " at entry " + std::to_string(i) + " out of [0, num_pages)");
    }
    for (int32_t n = 0; n < n_nodes; ++n) {
        if (T.len[n] < 0) return bad(PST_EINVAL, "tree_build: negative length at node " + std::to_string(n));
        if (T.parent[n] < -1 || T.parent[n] >= n_nodes)
            return bad(PST_ERANGE, "tree_build: parent out of range at node " + std::to_string(n));
        if (T.parent[n] == n) return bad(PST_ECYCLE, "tree_build: node " + std::to_string(n) + " is its own parent");
        const int32_t fo = T.first_offset[n];
        if (fo < 0 || fo >= page_size)
            return bad(PST_ERANGE, "tree_build: first_offset out of [0, page_size) at node " + std::to_string(n));
        const int64_t have = (page_ptr[n + 1] - page_ptr[n]) * (int64_t)page_size;
        if (T.len[n] > 0 && (int64_t)fo + T.len[n] > have)
            return bad(PST_ERANGE, "tree_build: node " + std::to_string(n) + " overruns its listed pages");
    }
    // children lists and cycle check (every walk to the top must end)
    T.children.assign(n_nodes, {});
    std::vector<int32_t> roots;
    for (int32_t n = 0; n < n_nodes; ++n) {
        if (T.parent[n] < 0) roots.push_back(n);
        else T.children[T.parent[n]].push_back(n);
    }
    T.depth.assign(n_nodes, -1);
    T.preorder.clear();
    T.preorder.reserve(n_nodes);
    std::vector<int32_t> stack;
    for (auto it = roots.rbegin(); it != roots.rend(); ++it) stack.push_back(*it);
    for (int32_t r : roots) T.depth[r] = 0;
    while (!stack.empty()) {
        int32_t n = stack.back();
        stack.pop_back();
        T.preorder.push_back(n);
        const auto& ch = T.children[n];
        for (auto it = ch.rbegin(); it != ch.rend(); ++it) {
            T.depth[*it] = T.depth[n] + 1;
            stack.push_back(*it);
        }
    }
    if ((int32_t)T.preorder.size() != n_nodes)
        return bad(PST_ECYCLE, "tree_build: parent array has a cycle (nodes unreachable from the virtual root)");
    T.unique_pages.assign(T.page_ids.begin(), T.page_ids.end());
    std::sort(T.unique_pages.begin(), T.unique_pages.end());
    T.unique_pages.erase(std::unique(T.unique_pages.begin(), T.unique_pages.end()), T.unique_pages.end());
    *out = t;
    return PST_OK;
}

extern "C" void pst_tree_destroy(pst_tree* t) { delete t; }
