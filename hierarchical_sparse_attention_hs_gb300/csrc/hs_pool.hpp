// Library-internal state of a pool, shared by the translation units of libhs.so (not part of the C ABI).
#ifndef HS_POOL_HPP_
#define HS_POOL_HPP_

#include <cstddef>
#include <cstdint>

#include "../../include/hs.h"

constexpr int HS_MAX_CLUSTER = 8;  // largest thread-block cluster a resolve launch uses

struct hs_pool {
  hs_pool_desc d;
  hs_meta_layout lay;
  int device;
  int num_sms;
  bool noio;
  const uint8_t* src;  // device-visible row source
  int32_t* step;
  int32_t* err;
  int32_t begin_pending;  // step increments deferred to the next resolve-type launch (hs_step_begin_fused)
  unsigned long long* counters;
  int32_t* tok2slot;
  int32_t* slot_tok;
  int32_t* slot_stamp;
  size_t smem;
  int max_cluster;   // largest cluster size that fits on the device for this shared-memory size
  int resident;      // resolve CTAs resident on the device at once (one wave)
  int max_active[HS_MAX_CLUSTER + 1];  // clusters of each size resident at once
};


#endif  // HS_POOL_HPP_
