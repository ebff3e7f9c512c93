// pages.cpp -- a host pool of KV pages with reference counts (deft_pages_*).
//
// DeFT Guide, "Production Engineering and Kernel Deployment Best
// Practices", items "Paged KV-Cache Compatibility" and "Tree Pruning Memory
// Management": the tree's KV lives in physical pages named through a page
// table, and the pages of branches that verification rejects go back to the
// pool at once, through reference counts, with no copying or compaction.
// The pool hands out page numbers only: the KV memory itself (k_pages /
// v_pages) is the caller's, and so is the page table the kernels read.
//
// Free pages are kept on a stack, so taking or returning a page is O(1).  A
// page may have several owners (a page table that shares it): each holds a
// reference, and the page is free again when the last is released.
#include <algorithm>
#include <cstdint>
#include <new>
#include <vector>

#include "deft.h"

struct deft_pages_t {
    std::vector<int32_t> ref;        // references per page (0: free)
    std::vector<int32_t> free_list;  // free pages, the next one to hand out last
};

namespace {

// Checks that `ids` are pages of the pool holding at least as many
// references as they appear times in `ids` (release) or at least one
// (retain).  `work` is scratch of the pool's size, left zeroed.
int check_ids(const deft_pages_t *pool, int32_t n, const int32_t *ids, bool releasing, std::vector<int32_t> &work)
{
    const int32_t np = (int32_t)pool->ref.size();
    int rc = DEFT_OK;
    int32_t i = 0;
    for (; i < n; ++i) {
        const int32_t p = ids[i];
        if (p < 0 || p >= np) {
            rc = DEFT_ERANGE;
            break;
        }
        if (pool->ref[p] - (releasing ? work[p] : 0) < 1) {
            rc = DEFT_ESTATE;   // a free page, or released more often than it is held
            break;
        }
        work[p] += 1;
    }
    for (int32_t j = 0; j < i; ++j)
        work[ids[j]] = 0;
    return rc;
}

}  // namespace

extern "C" {

int deft_pages_create(int32_t num_pages, deft_pages_t **out)
{
    if (!out)
        return DEFT_EINVAL;
    *out = nullptr;
    if (num_pages < 1)
        return DEFT_EINVAL;
    deft_pages_t *pool = new (std::nothrow) deft_pages_t();
    if (!pool)
        return DEFT_ENOMEM;
    try {
        pool->ref.assign(num_pages, 0);
        pool->free_list.resize(num_pages);
    } catch (const std::bad_alloc &) {
        delete pool;
        return DEFT_ENOMEM;
    }
    // Page 0 is handed out first.
    for (int32_t i = 0; i < num_pages; ++i)
        pool->free_list[i] = num_pages - 1 - i;
    *out = pool;
    return DEFT_OK;
}

void deft_pages_free(deft_pages_t *pool) { delete pool; }

int deft_pages_alloc(deft_pages_t *pool, int32_t n, int32_t *page_ids)
{
    if (!pool || n < 0 || (n > 0 && !page_ids))
        return DEFT_EINVAL;
    if ((size_t)n > pool->free_list.size())
        return DEFT_ENOMEM;   // nothing taken
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = pool->free_list.back();
        pool->free_list.pop_back();
        pool->ref[p] = 1;
        page_ids[i] = p;
    }
    return DEFT_OK;
}

int deft_pages_retain(deft_pages_t *pool, int32_t n, const int32_t *page_ids)
{
    if (!pool || n < 0 || (n > 0 && !page_ids))
        return DEFT_EINVAL;
    std::vector<int32_t> work;
    try {
        work.assign(pool->ref.size(), 0);
    } catch (const std::bad_alloc &) {
        return DEFT_ENOMEM;
    }
    const int rc = check_ids(pool, n, page_ids, false, work);
    if (rc != DEFT_OK)
        return rc;
    for (int32_t i = 0; i < n; ++i)
        pool->ref[page_ids[i]] += 1;
    return DEFT_OK;
}

int deft_pages_release(deft_pages_t *pool, int32_t n, const int32_t *page_ids)
{
    if (!pool || n < 0 || (n > 0 && !page_ids))
        return DEFT_EINVAL;
    std::vector<int32_t> work;
    try {
        work.assign(pool->ref.size(), 0);
    } catch (const std::bad_alloc &) {
        return DEFT_ENOMEM;
    }
    const int rc = check_ids(pool, n, page_ids, true, work);
    if (rc != DEFT_OK)
        return rc;   // nothing released
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = page_ids[i];
        if (--pool->ref[p] == 0)
            pool->free_list.push_back(p);
    }
    return DEFT_OK;
}

int32_t deft_pages_free_count(const deft_pages_t *pool)
{
    return pool ? (int32_t)pool->free_list.size() : -1;
}

int32_t deft_pages_refcount(const deft_pages_t *pool, int32_t page)
{
    if (!pool || page < 0 || page >= (int32_t)pool->ref.size())
        return -1;
    return pool->ref[page];
}

}  // extern "C"
