"""B300-native low-latency sum AllReduce over virtual ranks (C-ABI library
libllar.so plus a thin Python binding in `llar`).

Importing the package loads nothing; `tp_allreduce_persistent_b300.llar`
loads the compiled library on first use and raises if it is missing.
"""
