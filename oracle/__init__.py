"""CPU oracle for the RocketKV hot path -- test infrastructure, never imported by the product path."""
from . import rocketkv  # noqa: F401
