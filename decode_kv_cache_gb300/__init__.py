"""LongFlow fused decode step on GB300: a C-ABI library (liblongflow.so) of
hand-written sm_103a kernels and its thin Python binding."""
from .longflow import *  # noqa: F401,F403
from .longflow import __all__  # noqa: F401
