"""libdspark: GB300-native batched speculative verification and the
hardware-aware prefix scheduler of DSpark, and its drafter's sequential stage
with the Markov head, behind a C-ABI
(include/dspark.h). Python calls go through `binding` (ctypes, argument
marshalling only); `workloads` generates seeded synthetic inputs."""
from .binding import (DsparkError, ScheduleBuffers, VerifyBuffers, dspark_draft_markov,  # noqa: F401
                      dspark_schedule, dspark_verify, draft_workspace_bytes,
                      schedule_workspace_bytes, verify_workspace_bytes)
