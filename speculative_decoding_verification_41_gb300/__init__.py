"""libdspark: GB300-native batched speculative verification and the
hardware-aware prefix scheduler of DSpark, behind a two-call C-ABI
(include/dspark.h). Python calls go through `binding` (ctypes, argument
marshalling only); `workloads` generates seeded synthetic inputs."""
from .binding import (DsparkError, ScheduleBuffers, VerifyBuffers, dspark_schedule,  # noqa: F401
                      dspark_verify, schedule_workspace_bytes, verify_workspace_bytes)
