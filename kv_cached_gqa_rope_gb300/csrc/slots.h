// Host-side slot table of the shared KV cache: which request owns which cache
// row and how many tokens that row holds.  Internal to libkvgqa; the C ABI in
// api.cu wraps it.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": the
// continuous-batch scheduler owns the request-to-row map above the model
// primitives; it admits only at step boundaries, resets a row when its request
// ends (length, stop or cancel) and reuses the lowest free slot, while the
// shared cache allocation itself persists.
#pragma once

#include <cstdint>
#include <map>
#include <vector>

namespace kvgqa {

class SlotTable {
 public:
  enum Reason { kStop = 0, kLength = 1, kCancel = 2 };

  SlotTable(int num_slots, int max_seq) : max_seq_(max_seq), owner_(num_slots, -1), length_(num_slots, 0) {}

  int num_slots() const { return static_cast<int>(owner_.size()); }
  int max_seq() const { return max_seq_; }
  int active() const { return static_cast<int>(row_of_.size()); }

  // Lowest free row for `request`, whose first `prompt_len` tokens are (or are
  // about to be) in that row; -1 when every row is taken.  A request already
  // admitted keeps its row (returned again).
  int admit(int64_t request, int prompt_len) {
    auto it = row_of_.find(request);
    if (it != row_of_.end()) return it->second;
    for (int r = 0; r < num_slots(); ++r) {
      if (owner_[r] < 0) {
        owner_[r] = request;
        length_[r] = prompt_len;
        row_of_[request] = r;
        return r;
      }
    }
    return -1;
  }

  // Free the request's row (its bytes stay; the next owner overwrites them).
  bool release(int64_t request, Reason why) {
    auto it = row_of_.find(request);
    if (it == row_of_.end()) return false;
    owner_[it->second] = -1;
    length_[it->second] = 0;
    row_of_.erase(it);
    ++released_[why];
    return true;
  }

  int row(int64_t request) const {
    auto it = row_of_.find(request);
    return it == row_of_.end() ? -1 : it->second;
  }
  int length(int64_t request) const {
    const int r = row(request);
    return r < 0 ? -1 : length_[r];
  }
  long long released(Reason why) const { return released_[why]; }

  // One decode step for `requests` (in the caller's order): the token of
  // request i goes to position length and row of that request.  Writes
  // tokens / positions / rows into meta[0][i], meta[1][i], meta[2][i] of a
  // [3][capacity] array, then advances every length by one; a request whose
  // row is then full (length == max_seq) is released with reason kLength and
  // flagged in finished[i].  Returns the index of the first unknown or full
  // request, or -1 on success (nothing is changed on failure).
  int step(const int64_t* requests, const int32_t* tokens, int n, int32_t* meta, int capacity, uint8_t* finished) {
    for (int i = 0; i < n; ++i) {
      const int r = row(requests[i]);
      if (r < 0 || length_[r] >= max_seq_) return i;
      for (int j = 0; j < i; ++j)
        if (requests[j] == requests[i]) return i;  // one token per request per step
    }
    for (int i = 0; i < n; ++i) {
      const int r = row(requests[i]);
      meta[i] = tokens ? tokens[i] : 0;
      meta[capacity + i] = length_[r];
      meta[2 * capacity + i] = r;
    }
    for (int i = 0; i < n; ++i) {
      const int r = row(requests[i]);
      ++length_[r];
      const bool full = length_[r] >= max_seq_;
      if (finished) finished[i] = full ? 1 : 0;
      if (full) release(requests[i], kLength);
    }
    return -1;
  }

 private:
  int max_seq_;
  std::vector<int64_t> owner_;   // request owning each row, -1 when free
  std::vector<int> length_;      // tokens held by each row
  std::map<int64_t, int> row_of_;
  long long released_[3] = {0, 0, 0};
};

}  // namespace kvgqa
