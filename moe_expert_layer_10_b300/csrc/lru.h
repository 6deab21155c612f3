// Host-side shared LRU policy over whole (layer, expert) cache entries.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- decode uses one shared LRU expert cache across layers and tokens, entries are
// complete layer-expert pairs, and the cache follows routing instead of being frozen at
// startup; "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves
// Large MoE Models" -- recently routed experts stay in VRAM, misses are filled over PCIe.
//
// Slot rule (the pages are silent): a miss takes the lowest free slot; when none is free
// it takes the slot of the least recently used entry. O(1) touch and evict: an intrusive
// doubly-linked recency list over slots plus a key -> slot array. Decisions are planned
// first and committed only after the fill copy was enqueued, so a failed fill leaves the
// policy exactly as it was.
#pragma once

#include <cstdint>
#include <set>
#include <vector>

namespace moe {

class ExpertLru {
   public:
    enum Kind { kHit = 0, kFill = 1, kPrefetchFill = 2, kPrefetchHit = 3 };

    struct Plan {
        int kind;
        int key;     // layer * num_experts + expert
        int slot;    // slot holding the key after commit
        int victim;  // evicted key, or -1
    };

    ExpertLru() = default;
    ExpertLru(int capacity, int num_keys) { reset(capacity, num_keys); }

    void reset(int capacity, int num_keys) {
        cap_ = capacity;
        slot_of_.assign(num_keys, -1);
        key_in_.assign(capacity, -1);
        prev_.assign(capacity, -1);
        next_.assign(capacity, -1);
        head_ = tail_ = -1;
        free_.clear();
        for (int s = 0; s < capacity; ++s) free_.insert(s);
    }

    int capacity() const { return cap_; }
    int slot_of(int key) const { return slot_of_[key]; }
    int key_in(int slot) const { return key_in_[slot]; }

    Plan plan(int key, bool prefetch) const {
        Plan p{0, key, -1, -1};
        const int s = slot_of_[key];
        if (s >= 0) {
            p.kind = prefetch ? kPrefetchHit : kHit;
            p.slot = s;
            return p;
        }
        p.kind = prefetch ? kPrefetchFill : kFill;
        if (!free_.empty()) {
            p.slot = *free_.begin();
        } else {
            p.slot = tail_;
            p.victim = key_in_[tail_];
        }
        return p;
    }

    void commit(const Plan& p) {
        if (p.kind == kHit || p.kind == kPrefetchHit) {
            unlink(p.slot);
            push_front(p.slot);
            return;
        }
        if (p.victim >= 0) {
            unlink(p.slot);
            slot_of_[p.victim] = -1;
        } else {
            free_.erase(p.slot);
        }
        key_in_[p.slot] = p.key;
        slot_of_[p.key] = p.slot;
        push_front(p.slot);
    }

   private:
    void unlink(int s) {
        if (prev_[s] >= 0) next_[prev_[s]] = next_[s];
        else head_ = next_[s];
        if (next_[s] >= 0) prev_[next_[s]] = prev_[s];
        else tail_ = prev_[s];
        prev_[s] = next_[s] = -1;
    }
    void push_front(int s) {
        prev_[s] = -1;
        next_[s] = head_;
        if (head_ >= 0) prev_[head_] = s;
        head_ = s;
        if (tail_ < 0) tail_ = s;
    }

    int cap_ = 0;
    std::vector<int> slot_of_, key_in_, prev_, next_;
    int head_ = -1, tail_ = -1;  // most / least recently used slot
    std::set<int> free_;
};

}  // namespace moe
