"""shared_prefix_fan_gb300 -- shared-prefix fan-out attention on GB300 (sm_103a).

  binding    ctypes binding of libfanout.so (fanout_attn, fanout_fork, ...)
  build      builds libfanout.so in-tree with nvcc
  workloads  seeded synthetic inputs (shared with the test oracle)
"""
__all__ = ["binding", "build", "workloads"]
