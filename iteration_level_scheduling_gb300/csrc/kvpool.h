// Token-granular K/V reservation pool (host-side metadata only).
//
// Orca reserves, when a request is admitted, K/V space for the request's
// maximum length and frees it when the request finishes ("論文解説: Orca",
// scheduler algorithm; garden.houmin.site Orca notes, 3.1.1).  A reservation
// here is one contiguous range of slots, placed first-fit at the lowest free
// offset; a free merges the range with its free neighbours.  The placement is
// deterministic, so slot indices can be compared exactly with a reference.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <unordered_map>

namespace orca {

// Host-side fault injection for failure-detection tests: the environment
// variable ORCA_FAULT holds comma-separated "point:N" entries; an entry for
// `point` makes the N-th call of that operation fail.  Read when the object
// that owns the operation is created.  Returns N, or 0 for no fault.
inline int64_t fault_point(const char *point) {
    const char *v = std::getenv("ORCA_FAULT");
    const size_t len = std::strlen(point);
    while (v && *v) {
        if (std::strncmp(v, point, len) == 0 && v[len] == ':') return std::strtoll(v + len + 1, nullptr, 10);
        v = std::strchr(v, ',');
        if (v) ++v;
    }
    return 0;
}

class KVPool {
  public:
    explicit KVPool(int64_t slots) : slots_(slots), fail_at_(fault_point("kv_alloc")) {
        if (slots > 0) free_[0] = slots;
    }

    int64_t slots() const { return slots_; }
    int64_t reserved() const { return reserved_; }

    // Returns the offset, -1 if no free range is large enough (or the call is
    // the one ORCA_FAULT=kv_alloc:N picks), -2 if the arguments are invalid.
    int64_t alloc(int64_t id, int64_t n) {
        if (n <= 0 || owned_.count(id)) return -2;
        if (++calls_ == fail_at_) return -1;
        for (auto it = free_.begin(); it != free_.end(); ++it) {
            if (it->second < n) continue;
            int64_t off = it->first, len = it->second;
            free_.erase(it);
            if (len > n) free_[off + n] = len - n;
            owned_[id] = {off, n};
            reserved_ += n;
            return off;
        }
        return -1;
    }

    bool release(int64_t id) {
        auto o = owned_.find(id);
        if (o == owned_.end()) return false;
        int64_t off = o->second.first, len = o->second.second;
        owned_.erase(o);
        reserved_ -= len;
        auto next = free_.lower_bound(off);
        if (next != free_.end() && off + len == next->first) {
            len += next->second;
            next = free_.erase(next);
        }
        if (next != free_.begin()) {
            auto prev = std::prev(next);
            if (prev->first + prev->second == off) {
                prev->second += len;
                return true;
            }
        }
        free_[off] = len;
        return true;
    }

    // (offset, length) of a reservation; false if the id holds none.
    bool lookup(int64_t id, int64_t *off, int64_t *len) const {
        auto o = owned_.find(id);
        if (o == owned_.end()) return false;
        *off = o->second.first;
        *len = o->second.second;
        return true;
    }

  private:
    int64_t slots_;
    int64_t fail_at_ = 0, calls_ = 0;
    int64_t reserved_ = 0;
    std::map<int64_t, int64_t> free_;  // offset -> length, sorted, never adjacent
    std::unordered_map<int64_t, std::pair<int64_t, int64_t>> owned_;
};

}  // namespace orca
