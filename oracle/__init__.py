"""Float64 CPU oracle for linear cross-entropy.  Test infrastructure only: the product path never
imports it (see ``lce_ref`` for the definition it follows and the readings it takes)."""
from .lce_ref import *  # noqa: F401,F403
from .lce_ref import __all__  # noqa: F401
