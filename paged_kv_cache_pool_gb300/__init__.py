"""Shared-prefix paged decode attention for GB300 (sm_103a).

The library is libgk.so (C ABI in include/gk.h); ``binding`` exposes the same
``gk_*`` calls to Python and ``engine`` strings them into decode steps.
"""
from . import binding  # noqa: F401
from .binding import GkError  # noqa: F401
