// plan_cache.h -- bounded least-recently-used map from a layout key to its plan
// (host only; no CUDA).
//
// An RL training loop repacks every micro-batch, so the response offsets -- and
// with them the work lists -- change from call to call.  The cache keeps the
// plans of the `capacity` most recently used layouts; inserting one more hands
// the least recently used entry back to the caller, which releases its memory
// once the GPU no longer reads it.
#pragma once
#include <stddef.h>

#include <list>
#include <memory>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

namespace dkv {

template <class V>
class LruCache {
 public:
  explicit LruCache(size_t capacity) : capacity_(capacity < 1 ? 1 : capacity) {}

  // The entry of `key`, marked most recently used, or nullptr.
  V* find(const std::string& key) {
    auto it = index_.find(key);
    if (it == index_.end()) return nullptr;
    order_.splice(order_.begin(), order_, it->second);
    return it->second->second.get();
  }

  // Inserts (or replaces) the entry of `key` as the most recently used one.  Entries
  // pushed out -- the least recently used beyond the capacity, and a replaced value --
  // are appended to `evicted`.
  V* insert(const std::string& key, std::unique_ptr<V> value, std::vector<std::unique_ptr<V>>* evicted) {
    auto it = index_.find(key);
    if (it != index_.end()) {
      evicted->push_back(std::move(it->second->second));
      order_.erase(it->second);
      index_.erase(it);
    }
    order_.emplace_front(key, std::move(value));
    index_[key] = order_.begin();
    while (order_.size() > capacity_) {
      auto last = std::prev(order_.end());
      evicted->push_back(std::move(last->second));
      index_.erase(last->first);
      order_.erase(last);
    }
    return order_.front().second.get();
  }

  // Removes every entry, least recently used first, into `evicted`.
  void clear(std::vector<std::unique_ptr<V>>* evicted) {
    while (!order_.empty()) {
      auto last = std::prev(order_.end());
      evicted->push_back(std::move(last->second));
      index_.erase(last->first);
      order_.erase(last);
    }
  }

  size_t size() const { return order_.size(); }
  size_t capacity() const { return capacity_; }

  // Keys from the most to the least recently used.
  std::vector<std::string> keys() const {
    std::vector<std::string> k;
    for (const auto& e : order_) k.push_back(e.first);
    return k;
  }

 private:
  using Entry = std::pair<std::string, std::unique_ptr<V>>;
  size_t capacity_;
  std::list<Entry> order_;  // most recently used first
  std::unordered_map<std::string, typename std::list<Entry>::iterator> index_;
};

}  // namespace dkv
