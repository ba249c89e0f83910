// lfu.h -- the per-layer expert cache policy (host side).
//
// The pages give a 16-slot least-frequently-used expert cache per layer
// (devtrends page, section "Qual e il trucco principale dell'architettura";
// remio.ai page, section "Mac Gemma 4 26B entra nello spazio disponibile...").
// The tie rules are this library's reading:
//   * a step brings a request list (the distinct experts of the step, in first
//     appearance order);
//   * every requested expert already resident is a hit: its use count grows by
//     one and its last-use step becomes the current step;
//   * then each missing expert, in request order, takes the lowest-numbered empty
//     slot, or else evicts, among the slots whose expert is not requested in this
//     step, the one with the smallest (use count, last-use step, slot number); the
//     newcomer starts with count 1 and last use = the current step (an evicted
//     expert's count is forgotten);
//   * more distinct experts than slots is a capacity error and changes nothing.
#pragma once

#include <stdint.h>

#include <vector>

namespace moe {

class LfuPolicy {
public:
    LfuPolicy(int slots, int experts)
        : slots_(slots), experts_(experts), expert_(slots, -1), count_(slots, 0), last_(slots, 0),
          where_(experts, -1), wanted_(experts, 0) {}

    int slots() const { return slots_; }
    int experts() const { return experts_; }
    uint64_t hits() const { return hits_; }
    uint64_t misses() const { return misses_; }
    int64_t steps() const { return step_; }
    int expert_in(int s) const { return expert_[s]; }
    uint32_t count_of(int s) const { return count_[s]; }
    int64_t last_of(int s) const { return last_[s]; }
    int slot_of(int e) const { return where_[e]; }

    // 0 = ok, 1 = bad request (expert out of range or repeated), 3 = capacity.
    // slot_out[i] / hit_out[i] describe request i (either may be null).
    int step(const int32_t *req, int n, int32_t *slot_out, uint8_t *hit_out) {
        if (n < 0 || (n > 0 && !req)) return 1;
        int bad = 0;
        for (int i = 0; i < n && !bad; i++) {
            if (req[i] < 0 || req[i] >= experts_ || wanted_[req[i]]) bad = 1;
            else wanted_[req[i]] = 1;
        }
        if (bad || n > slots_) {
            for (int i = 0; i < n; i++)
                if (req[i] >= 0 && req[i] < experts_) wanted_[req[i]] = 0;
            return bad ? 1 : 3;
        }
        for (int i = 0; i < n; i++) {
            const int s = where_[req[i]];
            if (s >= 0) {
                count_[s]++;
                last_[s] = step_;
                hits_++;
            }
            if (hit_out) hit_out[i] = s >= 0;
            if (slot_out) slot_out[i] = s;
        }
        // requested experts are never evicted below, so where_ still tells hits apart
        for (int i = 0; i < n; i++) {
            const int e = req[i];
            if (where_[e] >= 0) continue;
            const int s = victim();
            if (expert_[s] >= 0) where_[expert_[s]] = -1;
            expert_[s] = e;
            where_[e] = s;
            count_[s] = 1;
            last_[s] = step_;
            misses_++;
            if (slot_out) slot_out[i] = s;
        }
        for (int i = 0; i < n; i++) wanted_[req[i]] = 0;
        step_++;
        return 0;
    }

    // Replaces the whole state (expert per slot with -1 = empty, counts, last uses,
    // the step counter and the running totals).
    void load(const int *expert_of, const uint32_t *count, const int64_t *last, int64_t step, uint64_t hits,
              uint64_t misses) {
        for (int e = 0; e < experts_; e++) where_[e] = -1;
        for (int s = 0; s < slots_; s++) {
            expert_[s] = expert_of[s];
            count_[s] = count[s];
            last_[s] = last[s];
            if (expert_[s] >= 0) where_[expert_[s]] = s;
        }
        step_ = step;
        hits_ = hits;
        misses_ = misses;
    }

    // Marks slot s empty (its contents are no longer known): the expert it held,
    // if any, is no longer resident.  Counts and totals are otherwise unchanged.
    void invalidate(int s) {
        if (s < 0 || s >= slots_ || expert_[s] < 0) return;
        where_[expert_[s]] = -1;
        expert_[s] = -1;
        count_[s] = 0;
        last_[s] = 0;
    }

private:
    int victim() const {
        for (int s = 0; s < slots_; s++)
            if (expert_[s] < 0) return s;
        int best = -1;
        for (int s = 0; s < slots_; s++) {
            if (wanted_[expert_[s]]) continue;
            if (best < 0 || count_[s] < count_[best] || (count_[s] == count_[best] && last_[s] < last_[best]))
                best = s;
        }
        return best;
    }

    int slots_, experts_;
    std::vector<int> expert_;      // expert held by each slot, -1 = empty
    std::vector<uint32_t> count_;  // uses since the expert entered its slot
    std::vector<int64_t> last_;    // step of the last use
    std::vector<int> where_;       // slot of each expert, -1 = not resident
    std::vector<unsigned char> wanted_;
    int64_t step_ = 0;
    uint64_t hits_ = 0, misses_ = 0;
};

}  // namespace moe
