"""fp64 CPU oracle for the ISD verify-and-propose step (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg import this package.  The product library never does.

``oracle.<name>`` calls go to the default build (oracle/liboracle.so);
``oracle.Oracle(path)`` loads another build of the same source.
"""
from .oracle import (DTYPE_BF16, DTYPE_F32, TAG_ACCEPT, TAG_BONUS, TAG_CORRECT,  # noqa: F401
                     TAG_PROPOSE, Oracle, default)


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(default(), name)
