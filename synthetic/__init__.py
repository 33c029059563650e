"""Seeded synthetic inputs shared by the tests and the bench (no optimizer arithmetic)."""

from . import configs, generators  # noqa: F401
