"""GB300-native MoE route-sort (placeholder; the CUDA binding is added with the library)."""
from . import datagen  # noqa: F401
