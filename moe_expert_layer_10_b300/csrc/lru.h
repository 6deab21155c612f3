// Host-side shared LRU policy over whole (layer, expert) cache entries.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- decode uses one shared LRU expert cache across layers and tokens, entries are
// complete layer-expert pairs, and the cache follows routing instead of being frozen at
// startup; "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves
// Large MoE Models" -- recently routed experts stay in VRAM, misses are filled over PCIe.
//
// Slot rule (the pages are silent): a miss takes the lowest free slot; when none is free
// it takes the slot of the least recently used entry. A capacity change (elastic cache)
// keeps the most recently used entries that fit, evicts the others least recent first, and
// renumbers the survivors 0, 1, ... in the order of their old slots, so the used slots are
// always 0 .. n_used-1 (release_slot, for a fill that failed after its copy was enqueued, is
// the one operation that frees a slot in the middle). O(1) touch and evict: an intrusive
// doubly-linked recency list over slots plus a key -> slot array. Decisions are planned
// first and committed only after the fill copy was enqueued, so a failed fill leaves the
// policy exactly as it was.
#pragma once

#include <algorithm>
#include <cstdint>
#include <set>
#include <utility>
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
    int used() const { return cap_ - static_cast<int>(free_.size()); }

    // Change the capacity. evicted receives (key, old slot) of each evicted entry, least
    // recent first; moved receives (old slot, new slot) of each survivor whose slot changes.
    void resize(int new_cap, std::vector<std::pair<int, int>>* evicted, std::vector<std::pair<int, int>>* moved) {
        std::vector<int> rec;  // used slots, most recent first
        for (int s = head_; s >= 0; s = next_[s]) rec.push_back(s);
        const int keep = std::min(static_cast<int>(rec.size()), new_cap);
        for (int i = static_cast<int>(rec.size()) - 1; i >= keep; --i) {
            evicted->push_back({key_in_[rec[i]], rec[i]});
            slot_of_[key_in_[rec[i]]] = -1;
        }
        std::vector<int> by_slot(rec.begin(), rec.begin() + keep);
        std::sort(by_slot.begin(), by_slot.end());
        std::vector<int> new_of(cap_, -1);
        for (int r = 0; r < keep; ++r) {
            new_of[by_slot[r]] = r;
            if (by_slot[r] != r) moved->push_back({by_slot[r], r});
        }
        std::vector<int> key2(new_cap, -1), prev2(new_cap, -1), next2(new_cap, -1);
        for (int r = 0; r < keep; ++r) key2[r] = key_in_[by_slot[r]];
        for (int i = 0; i < keep; ++i) {
            const int s = new_of[rec[i]];
            prev2[s] = i > 0 ? new_of[rec[i - 1]] : -1;
            next2[s] = i + 1 < keep ? new_of[rec[i + 1]] : -1;
        }
        head_ = keep > 0 ? new_of[rec[0]] : -1;
        tail_ = keep > 0 ? new_of[rec[keep - 1]] : -1;
        for (int r = 0; r < keep; ++r) slot_of_[key2[r]] = r;
        key_in_.swap(key2);
        prev_.swap(prev2);
        next_.swap(next2);
        cap_ = new_cap;
        free_.clear();
        for (int s2 = keep; s2 < new_cap; ++s2) free_.insert(s2);
    }

    // The recency list and slot contents, for a policy that runs elsewhere (the GPU).
    void export_state(std::vector<int>* prev, std::vector<int>* next, std::vector<int>* key, int* head, int* tail,
                      int* n_used) const {
        *prev = prev_;
        *next = next_;
        *key = key_in_;
        *head = head_;
        *tail = tail_;
        *n_used = used();
    }
    void import_state(const std::vector<int>& prev, const std::vector<int>& next, const std::vector<int>& key,
                      int head, int tail, int n_used) {
        prev_ = prev;
        next_ = next;
        key_in_ = key;
        head_ = head;
        tail_ = tail;
        std::fill(slot_of_.begin(), slot_of_.end(), -1);
        for (int s = 0; s < cap_; ++s)
            if (key_in_[s] >= 0) slot_of_[key_in_[s]] = s;
        free_.clear();
        for (int s = n_used; s < cap_; ++s) free_.insert(s);
    }
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

    // Forget the entry in `slot` (if any) and return the slot to the free set: used when a
    // fill copy into the slot was enqueued but the fill could not be completed, so the slot
    // holds neither its old entry nor a usable new one.
    void release_slot(int slot) {
        const int key = key_in_[slot];
        if (key < 0) return;
        unlink(slot);
        slot_of_[key] = -1;
        key_in_[slot] = -1;
        free_.insert(slot);
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
