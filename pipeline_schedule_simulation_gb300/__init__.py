"""GB300-native batched evaluator of pipeline-parallel training schedules.

GPipe (and its first-in-first-out variant), synchronous 1F1B (PipeDream-Flush),
interleaved 1F1B and the Zero Bubble schedules ZB1P / ZB2P: per-device op
order, every op's start/end tick by max-plus longest path, makespan, per-stage
busy/idle ticks, the exact bubble fraction and the peak count of held
activations, for thousands to millions of instances per call; plus GPU
searches over contiguous layer-to-stage partitions (seeded, exhaustive, and
interleaved layouts).

The compute runs in hand-written CUDA kernels behind the C ABI declared in
``include/ppsched.h`` (``libppsched.so``); ``binding`` marshals arguments only.
Importing this package does not load the library: ``binding`` does, and fails
loudly if it has not been built.
"""
__all__ = ["binding", "workloads", "sharding", "timeline"]
