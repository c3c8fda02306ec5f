"""CPU oracle for the UFP4 hot path -- test infrastructure, not the library.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package.
"""
