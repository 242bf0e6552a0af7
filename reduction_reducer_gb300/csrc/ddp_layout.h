// Read-only access to a context's bucket layout from other translation units
// of the library (not part of the public ABI).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "ddp_reducer.h"

namespace ddp_internal {

struct Layout {
    int32_t P = 0;
    int32_t B = 0;
    int elem = 4;                                    // gradient element size in bytes
    bool bf16 = false;
    const int64_t* numel = nullptr;                  // [P]
    const ddp_locator* loc = nullptr;                // [P]
    const int64_t* bucket_off = nullptr;             // [B+1]
    const std::vector<std::vector<int32_t>>* members = nullptr;   // per bucket, push order
};

Layout layout(const ddp_ctx* ctx);

// Record the detail returned by ddp_last_error(ctx).
void set_error(ddp_ctx* ctx, const std::string& msg);

}  // namespace ddp_internal
