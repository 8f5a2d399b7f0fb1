"""CPU oracle for the KVMem decode hot path (test infrastructure only).

Imported by tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline
and reference legs; never by the product package.
"""
from . import kvm_oracle  # noqa: F401
