"""GB300-native (sm_103a) paged MLA decode.

The compute path lives in the C ABI library ``lib/libmla_decode.so`` built
from ``csrc/`` (see ``build.py``); ``mla`` is its Python binding.
"""
from .mla import (MLADecoder, MLAError, mla_decode_plan, mla_decode_run,  # noqa: F401
                  mla_decode_run_host, mla_plan_check_status, mla_plan_create,
                  mla_plan_destroy, mla_plan_info, mla_plan_partition_host)
