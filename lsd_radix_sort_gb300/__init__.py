"""GB300-native LSD radix sort (placeholder; the binding is added with the library)."""
