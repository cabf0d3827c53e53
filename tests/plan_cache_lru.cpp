// Host check of the plan cache's eviction order (compiled and run by
// tests/test_host_abi.py::test_plan_cache_evicts_least_recently_used).
#include <cstdio>
#include <memory>
#include <string>
#include <vector>

#include "plan_cache.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("FAILED line %d: %s\n", __LINE__, #c);      \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  dkv::LruCache<int> c(3);
  std::vector<std::unique_ptr<int>> ev;
  c.insert("a", std::unique_ptr<int>(new int(1)), &ev);
  c.insert("b", std::unique_ptr<int>(new int(2)), &ev);
  c.insert("c", std::unique_ptr<int>(new int(3)), &ev);
  CHECK(ev.empty() && c.size() == 3);
  CHECK(c.find("a") && *c.find("a") == 1);  // a becomes most recently used: order a, c, b
  c.insert("d", std::unique_ptr<int>(new int(4)), &ev);
  CHECK(ev.size() == 1 && *ev[0] == 2);      // b was the least recently used
  CHECK(!c.find("b") && c.size() == 3);
  CHECK((c.keys() == std::vector<std::string>{"d", "a", "c"}));
  ev.clear();
  c.insert("a", std::unique_ptr<int>(new int(5)), &ev);  // replacing hands back the old value
  CHECK(ev.size() == 1 && *ev[0] == 1 && *c.find("a") == 5 && c.size() == 3);
  ev.clear();
  for (int i = 0; i < 100; ++i) c.insert("k" + std::to_string(i), std::unique_ptr<int>(new int(i)), &ev);
  CHECK(c.size() == 3 && ev.size() == 100);  // 3 old entries + 97 of the new ones pushed out
  CHECK((c.keys() == std::vector<std::string>{"k99", "k98", "k97"}));
  ev.clear();
  c.clear(&ev);
  CHECK(c.size() == 0 && ev.size() == 3 && *ev[0] == 97 && *ev[2] == 99);  // least recently used first
  dkv::LruCache<int> one(0);  // capacity is at least one
  one.insert("x", std::unique_ptr<int>(new int(7)), &ev);
  CHECK(one.size() == 1 && one.capacity() == 1);
  std::printf("ok\n");
  return 0;
}
