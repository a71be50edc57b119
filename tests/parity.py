"""The parity rules (oracle/parity.py) and the workloads' device copies
(workloads/device.py), under the names the tests use."""
from oracle.parity import *  # noqa: F401,F403
from oracle.parity import ATTN_U, TOL, attention_reference, check_rule_a, check_rule_b, check_rule_c, \
    check_rule_d, rule_c, score_errors  # noqa: F401
from workloads.device import attn_to_device, to_device  # noqa: F401
