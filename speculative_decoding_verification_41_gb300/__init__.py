"""libdspark: GB300-native batched speculative verification and the
confidence-driven prefix scheduler of DSpark, behind a two-call C-ABI."""
