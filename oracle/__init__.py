"""CPU oracle (test infrastructure only; the library never imports it)."""

from . import vbq_oracle  # noqa: F401
