"""Host-side workload generation: the physical block allocator and the
continuous-batching step driver.  Pure Python; no GPU work happens here."""
from .allocator import BlockAllocator, OutOfBlocks
from .trace import CONTINUOUS_BATCHING_TRACE, ContinuousBatchingTrace, StepPlan, TraceConfig

__all__ = ["BlockAllocator", "OutOfBlocks", "ContinuousBatchingTrace", "StepPlan", "TraceConfig",
           "CONTINUOUS_BATCHING_TRACE"]
