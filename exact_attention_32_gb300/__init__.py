"""GB300-native exact attention forward (sm_103a)."""
from .workloads import HEADLINE, WORKLOADS, Workload, make_inputs, workload_inputs  # noqa: F401
