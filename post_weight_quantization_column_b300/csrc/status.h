// Device-side status codes: the same numbers as the public awq_status enum.
#pragma once
#include "../../include/awq.h"

#define AWQ_DEV_RANGE ((uint32_t)AWQ_ERR_RANGE)
#define AWQ_DEV_NONFINITE ((uint32_t)AWQ_ERR_NONFINITE)
#define AWQ_DEV_TIMEOUT ((uint32_t)AWQ_ERR_TIMEOUT)
